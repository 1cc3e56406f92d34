/*
 * cpattn - packed variable-length context-parallel attention on one GB300.
 *
 * C ABI of libcpattn.so.  Plain pointers and sizes only.
 *
 * Problem statement followed by this library:
 *   - Packed THD inputs: variable-length sequences concatenated along T and
 *     described by cu_seqlens ("Speeding up Variable-Length Training with
 *     Dynamic Context Parallelism and NVIDIA Megatron Core", section on
 *     dynamic rescheduling and packing, Fig. 1; PackedSeqParams carries
 *     cu_seqlens and cp_size).
 *   - A context-parallel (CP) group splits one sequence across ranks and runs
 *     blockwise attention while KV blocks circulate in a ring ("Scaling video
 *     training with parallelism", section 2, Ring Attention); the split is the
 *     load-balanced zigzag of ZIGZAG-RINGATTN (LongVILA news article, Fig. 5,
 *     Table 2) or a 2-D h x w tile grid (LongCat-Video context-parallel
 *     article, tensor split strategy: split_tensor_in_cp_2d,
 *     get_optimal_split, split_cp_2d / gather_cp_2d).
 *   - Splitting must not change what the model computes ("Scaling video
 *     training with parallelism", opening section): the merged result equals
 *     plain softmax attention inside each packed sequence.
 *   - Loss is normalised per valid token and FLOPs are counted from the real
 *     sequence lengths (Dynamic-CP article, section "Loss computation and
 *     FLOPS statistics").
 * Every virtual CP rank is emulated on the one GPU: a ring step is a change
 * of which KV rows a thread block reads next; no collective is issued.
 *
 * Conventions
 *   - Layouts (row-major, contiguous):  Q [T,H,D], K and V [T,Hkv,D],
 *     O [T,H,D] in the input dtype, LSE [H,T] fp32 (natural log, scale
 *     included).  Query head h reads KV head floor(h*Hkv/H).
 *   - Supported: dtype fp32 or bf16, D in {64, 128}, H % Hkv == 0,
 *     1 <= H, Hkv <= 256, T < 2^31.  Anything else: CPATTN_UNSUPPORTED or
 *     CPATTN_INVALID_ARG.  Device buffers must be 16-byte aligned.
 *   - Every function returns a status and never aborts or exits.  The
 *     message of the last failure on the calling thread is
 *     cpattn_last_error_string().
 *   - Device pointers are owned by the caller.  The library allocates no
 *     device memory: functions that need scratch take a caller-provided
 *     workspace of at least cpattn_workspace_size() bytes (256-byte aligned).
 *     Plans are host objects owned by the library, freed with
 *     cpattn_plan_destroy().
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Device work
 *     is asynchronous; argument errors are reported synchronously.  Every
 *     wait inside a kernel is bounded: one that runs out records a fault in
 *     the workspace and the kernel returns early; cpattn_sync_status()
 *     reports it as CPATTN_DEVICE_FAULT.
 */
#ifndef CPATTN_H
#define CPATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum cpattn_status {
  CPATTN_OK = 0,
  CPATTN_INVALID_ARG = 1,   /* bad pointer, size, cu_seqlens or plan input   */
  CPATTN_UNSUPPORTED = 2,   /* valid request this build does not implement   */
  CPATTN_WORKSPACE = 3,     /* workspace missing, misaligned or too small    */
  CPATTN_CUDA_ERROR = 4,    /* a CUDA runtime/driver call failed             */
  CPATTN_DEVICE_FAULT = 5   /* a kernel recorded a fault in the workspace    */
} cpattn_status_t;

typedef enum cpattn_mode {
  CPATTN_MODE_ZIGZAG = 0,      /* 2*cp chunks per sequence, rank r owns r and 2cp-1-r */
  CPATTN_MODE_GRID2D = 1,      /* one F x h x w latent cut into split_h x split_w tiles */
  CPATTN_MODE_CONTIGUOUS = 2,  /* packed T cut into cp contiguous ranges              */
  CPATTN_MODE_ULYSSES2D = 3,   /* u x r mesh: Ulysses all-to-all x zigzag ring (cpattn_plan_2d) */
  CPATTN_MODE_PAIRED = 4       /* clean/noisy time-chunk pairs, teacher forcing (cpattn_plan_paired) */
} cpattn_mode_t;

typedef enum cpattn_dtype {
  CPATTN_DTYPE_FP32 = 0,
  CPATTN_DTYPE_BF16 = 1
} cpattn_dtype_t;

/* Which part of a (q rank, ring step) pair can interact under a causal mask. */
typedef enum cpattn_mask_kind {
  CPATTN_MASK_SKIP = 0,     /* nothing visible                                   */
  CPATTN_MASK_FULL = 1,     /* every allowed pair (no causal cut inside the pair) */
  CPATTN_MASK_DIAG = 2,     /* the rank's own shard: causal inside               */
  CPATTN_MASK_KV_HEAD = 3,  /* zigzag, kv rank < q rank: the kv rank's first chunk only */
  CPATTN_MASK_Q_TAIL = 4    /* zigzag, kv rank > q rank: the q rank's second chunk only */
} cpattn_mask_kind_t;

typedef struct cpattn_grid {
  int32_t frames, height, width;   /* latent grid, tokens flattened (f, y, x) row-major */
} cpattn_grid_t;

typedef struct cpattn_plan cpattn_plan_t;

typedef struct cpattn_plan_info {
  int64_t total_tokens;     /* T = cu_seqlens[n_seqs]                            */
  int64_t n_chunks;         /* contiguous global row runs the split cuts T into  */
  int64_t max_rank_tokens;  /* largest per-rank shard                            */
  int32_t n_seqs;
  int32_t cp_size;
  int32_t mode;             /* cpattn_mode_t                                     */
  int32_t split_h;          /* GRID2D: tiles per column; ULYSSES2D: u; PAIRED: cp; else 0 */
  int32_t split_w;          /* GRID2D: tiles per row; ULYSSES2D: r; PAIRED: 1; else 0     */
  int32_t reserved;
} cpattn_plan_info_t;

/* ---------------------------------------------------------------- planning */

/* Build the context-parallel split of a packed batch for `cp_size` virtual
 * ranks.  Integer-only and deterministic.
 *   cu_seqlens_host: host int32 [n_seqs+1], cu[0] = 0, strictly increasing.
 *   ZIGZAG: sequence s (length L >= 2*cp) is cut into C = 2*cp chunks of
 *     floor(L/C) + [j < L mod C] tokens; rank r owns chunks r and C-1-r
 *     (zigzag ring split: LongVILA news article, Fig. 5 / Table 2).
 *   GRID2D: n_seqs must be 1 and grid F*h*w must equal T.  (split_h, split_w)
 *     is the factor pair of cp closest to square, the larger factor on the
 *     larger side (tie: split_h <= split_w); sides are cut in pieces of
 *     ceil(n/parts) with the remainder last; rank = ih*split_w + iw
 *     (LongCat-Video article, tensor split strategy, get_optimal_split).
 *   CONTIGUOUS: T cut into cp ranges, the first T mod cp one token longer
 *     (token stage of MM-SP: "Scaling video training with parallelism",
 *     section 3, Fig. 2).
 *   grid: required for GRID2D, ignored otherwise (may be NULL).
 *   out_plan: receives a plan owned by the caller until cpattn_plan_destroy.
 * Errors: CPATTN_INVALID_ARG for cp_size < 1, bad cu_seqlens, a zigzag
 * sequence shorter than 2*cp, a grid that does not match T or cannot be cut
 * into the required pieces, or fewer tokens than ranks. */
cpattn_status_t cpattn_plan(const int32_t* cu_seqlens_host, int32_t n_seqs, int32_t cp_size,
                            cpattn_mode_t mode, const cpattn_grid_t* grid,
                            cpattn_plan_t** out_plan);

/* The 2D-Attention mesh of ulysses x ring virtual ranks (LongVILA news
 * article, 2D attention parallelism and Fig. 3 left: independent Ulysses
 * all-to-all groups and Ring P2P groups, e.g. 8-way SP as a 4 x 2 mesh; USP
 * and LoongTrain: "Scaling video training with parallelism", section 2).
 * Mode CPATTN_MODE_ULYSSES2D, cp = ulysses * ring, rank g = j*ulysses + i
 * (i: position in its Ulysses group, j: ring index).
 *   Sequence-sharded layout (before the all-to-all): ring shard j is the
 *   zigzag split over `ring` (chunks j and 2*ring-1-j of every sequence, each
 *   sequence at least 2*ring tokens); its local rows are cut into `ulysses`
 *   contiguous pieces of floor(T_j/u) + [i < T_j mod u] rows, piece i going to
 *   rank (i, j).  rank_offsets / index_map / local_cu_seqlens describe this
 *   layout; chunks are the maximal runs of consecutive global rows of one
 *   sequence owned by one rank.
 *   After the all-to-all (cpattn_plan_get_a2a_map) rank (i, j) holds every row
 *   of ring shard j for query heads [i*H/u, (i+1)*H/u) and KV heads
 *   [i*Hkv/u, (i+1)*Hkv/u); the ring then runs over the r ring groups.
 * Errors: as cpattn_plan; ulysses, ring >= 1. */
cpattn_status_t cpattn_plan_2d(const int32_t* cu_seqlens_host, int32_t n_seqs, int32_t ulysses, int32_t ring,
                               cpattn_plan_t** out_plan);

/* LongLive-2.0's balanced SP for autoregressive teacher forcing ("Scaling
 * video training with parallelism", section 4): each sample of L tokens (L
 * even) is [clean history ; noisy target], each stream cut into n_chunks time
 * chunks of floor((L/2)/N) + [j < (L/2) mod N] tokens (at least one each).
 * Rank k keeps time chunks [k*m, (k+1)*m) (m = n_chunks / cp_size, which must
 * be an integer), each as its clean chunk then its noisy chunk; the forward
 * runs behind a Ulysses all-to-all over all cp ranks (split_h = cp, split_w =
 * 1, cpattn_plan_get_a2a_map) with the teacher-forcing mask in that order:
 * a clean token of chunk j sees the clean tokens of chunks <= j, a noisy token
 * of chunk j the clean tokens of chunks < j and the noisy tokens of chunk j
 * (the page is cut off before it states the mask; this is the reading used).
 * Chunks are listed clean chunks first, then noisy chunks, per sample.
 * cpattn_fwd needs causal = 1 (the teacher-forcing mask) and H, Hkv multiples
 * of cp.  Errors: as cpattn_plan. */
cpattn_status_t cpattn_plan_paired(const int32_t* cu_seqlens_host, int32_t n_seqs, int32_t cp_size,
                                   int32_t n_chunks, cpattn_plan_t** out_plan);

/* Number of (query, key) pairs that a plan's mask allows: per sequence
 * L(L+1)/2 (causal) or L^2, or the teacher-forcing count of a PAIRED plan.
 * Forward FLOPs = 4 * D * H * pairs. */
cpattn_status_t cpattn_plan_allowed_pairs(const cpattn_plan_t* plan, int32_t causal, uint64_t* out);

/* Free a plan (NULL is a no-op). */
cpattn_status_t cpattn_plan_destroy(cpattn_plan_t* plan);

/* Summary sizes of a plan. */
cpattn_status_t cpattn_plan_get_info(const cpattn_plan_t* plan, cpattn_plan_info_t* out);

/* Host copies of the plan's integer maps.  `n` is the capacity of `out` in
 * elements; CPATTN_INVALID_ARG if it is smaller than required.
 *   chunk_offsets [n_chunks+1]: global start row of each chunk, then T.
 *     ZIGZAG chunk (s, j) is entry s*2cp + j; GRID2D chunks are the
 *     (frame, row, w-piece) runs in global order; CONTIGUOUS chunk r is rank r.
 *   chunk_ranks [n_chunks]: owning rank of each chunk.
 *   rank_offsets [cp+1]: start of each rank's rows in the index map.
 *   local_cu_seqlens [n_seqs+1] for `rank`: the rank's local rows per sequence.
 *   index_map [T]: rank-major local row -> global row (zigzag local order is
 *     chunk r then chunk 2cp-1-r of each sequence; grid tiles are (f, y, x)
 *     row-major).
 *   ring schedule [cp*cp] at index r*cp + t: the kv rank that q rank r works
 *     with at ring step t, (r - t) mod cp ("Scaling video training with
 *     parallelism", section 2, Ring Attention), and its cpattn_mask_kind_t
 *     under `causal` (causal GRID2D plans: CPATTN_UNSUPPORTED). */
cpattn_status_t cpattn_plan_get_chunk_offsets(const cpattn_plan_t* plan, int64_t* out, int64_t n);
cpattn_status_t cpattn_plan_get_chunk_ranks(const cpattn_plan_t* plan, int32_t* out, int64_t n);
cpattn_status_t cpattn_plan_get_rank_offsets(const cpattn_plan_t* plan, int64_t* out, int64_t n);
cpattn_status_t cpattn_plan_get_local_cu_seqlens(const cpattn_plan_t* plan, int32_t rank,
                                                 int32_t* out, int64_t n);
cpattn_status_t cpattn_plan_get_index_map(const cpattn_plan_t* plan, int64_t* out, int64_t n);
cpattn_status_t cpattn_plan_get_ring_schedule(const cpattn_plan_t* plan, int32_t causal,
                                              int32_t* kv_rank, int32_t* mask_kind, int64_t n);

/* ULYSSES2D and PAIRED plans: the all-to-all as one row gather.  Viewing a [T,H,D]
 * tensor as [T*u, H/u*D] rows (row t*u + i = token t's head group i), row
 * i*T + p of the head-sharded buffer is source row out[i*T + p] =
 * index_map[p]*u + i: head group i's rows are the ring shards in ring order,
 * each in its zigzag local order.  `out` is host int64 [u*T].  The ring
 * schedule of these plans has (i, j) at step t < r working with the ring
 * shard of rank ((j - t) mod r)*u + i, and kv rank -1 (SKIP) for t >= r.
 * Other plans: CPATTN_INVALID_ARG. */
cpattn_status_t cpattn_plan_get_a2a_map(const cpattn_plan_t* plan, int64_t* out, int64_t n);

/* The work list a call hands its kernel, as a host copy (so the planner can
 * be checked against the mask's definition without a GPU).
 *   backward = 0: the query tiles of cpattn_fwd (q_rank = -1) or of
 *     cpattn_block_fwd(q_rank, ring_step), each with the key runs it reads,
 *     in ring order (at step t the queries of rank r read the KV shard of
 *     rank (r - t) mod cp).
 *   backward = 1: the key tiles of cpattn_bwd / cpattn_block_bwd, each with
 *     the query runs that see it, in ring order (the KV shard of rank k
 *     meets the queries of rank (k + t) mod cp at step t).
 * Tile and piece sizes are those of the kernel for `dtype`.
 *   tile: row0, pos0, rows = its rows (buffer row, position inside the
 *     sequence (GRID2D, bidirectional only: the gathered row), count);
 *     out_row0 = output row of the first; runs
 *     [run_begin, run_end); pieces = kernel loop trips over its runs; rank =
 *     the virtual rank that owns the tile.  A tile of one ring step lies in
 *     one chunk of its rank.  A tile of a whole forward call on global rows
 *     (zigzag, contiguous) is cut from its sequence, ending at the
 *     sequence's last row, up to the kernel's tile height, so it may hold
 *     the end of one chunk and the start of the next; its rank owns its last
 *     row and its runs follow that rank's ring, with the position mask in
 *     every run that crosses the tile's first query.  A key tile of a whole
 *     backward call on global rows is cut from its sequence's first row on;
 *     its rank owns its first key and its query runs follow that rank's
 *     ring.  Runs of one ring step that continue each other are merged.
 *   run: row0, pos0, len = rows of the other side; masked = 1 when the
 *     position mask (key position <= query position) applies inside the run,
 *     0 when every pair of the tile and the run is allowed.
 * Rows are rows of the buffers the kernel reads: global rows, for GRID2D the
 * gathered rank-major rows of the index map, for ULYSSES2D and PAIRED the
 * rows of the head-sharded buffers (head group i at i*T).  *n_tiles and
 * *n_runs receive the counts; tiles and runs (capacities max_tiles,
 * max_runs) may be NULL to ask for the counts only.  Errors: those of the
 * call described (unsupported plan, mode or causal flag, rank or step out of
 * range); CPATTN_INVALID_ARG when a buffer is smaller than its count. */
typedef struct cpattn_work_tile_t {
  int32_t row0, pos0, out_row0, rows, run_begin, run_end, pieces, rank;
} cpattn_work_tile_t;
typedef struct cpattn_work_run_t {
  int32_t row0, pos0, len, masked;
} cpattn_work_run_t;
cpattn_status_t cpattn_plan_get_worklist(const cpattn_plan_t* plan, int32_t backward, cpattn_dtype_t dtype,
                                         int32_t causal, int32_t q_rank, int32_t ring_step,
                                         cpattn_work_tile_t* tiles, int64_t max_tiles, cpattn_work_run_t* runs,
                                         int64_t max_runs, int64_t* n_tiles, int64_t* n_runs);

/* ---------------------------------------------------------------- attention */

/* Bytes of device workspace that cpattn_fwd / cpattn_block_fwd need for this
 * plan and shape (work list, fault word and, for GRID2D, the gathered
 * shards; for ULYSSES2D, the all-to-all map and head-sharded buffers). */
cpattn_status_t cpattn_workspace_size(const cpattn_plan_t* plan, int32_t H, int32_t Hkv, int32_t D,
                                      cpattn_dtype_t dtype, int32_t causal, size_t* bytes);

/* Whole packed forward: every virtual rank's query shard attends, ring step
 * by ring step, to the KV shard it holds at that step; each step's partial is
 * merged into the running result by exact log-sum-exp rescaling, and the
 * final O/LSE are written at global THD rows.  Equals plain softmax attention
 * inside each packed sequence (causal: key position <= query position).
 *   q, k, v: device, layouts above, dtype `dtype`.
 *   scale:   softmax scale (commonly 1/sqrt(D)).
 *   o:       device [T,H,D] dtype;  lse: device [H,T] fp32.
 *   workspace/ws_bytes: device scratch, >= cpattn_workspace_size().
 * GRID2D gathers each rank's shard into the workspace first (split_cp_2d)
 * and writes outputs back through the index map (gather_cp_2d).
 * Causal GRID2D is CPATTN_UNSUPPORTED.
 * ULYSSES2D performs the all-to-all (a row gather of Q, K, V into
 * head-sharded buffers in the workspace), runs every head group's ring over
 * the r ring shards in one launch, then the reverse all-to-all of O and LSE;
 * H and Hkv must be multiples of u (else CPATTN_UNSUPPORTED).
 * PAIRED plans take the same path with the teacher-forcing mask (causal = 1).
 * cpattn_block_fwd, cpattn_bwd, cpattn_block_bwd and cpattn_fwd_static
 * return CPATTN_UNSUPPORTED for ULYSSES2D and PAIRED plans. */
cpattn_status_t cpattn_fwd(const cpattn_plan_t* plan, const void* q, const void* k, const void* v,
                           cpattn_dtype_t dtype, int32_t H, int32_t Hkv, int32_t D, float scale,
                           int32_t causal, void* o, float* lse, void* workspace, size_t ws_bytes,
                           void* stream);

/* One ring step of one virtual rank: the attention of rank `q_rank`'s query
 * shard over the KV shard of rank (q_rank - ring_step) mod cp, as a partial
 * result normalised over that block ("Scaling video training with
 * parallelism", section 2, Ring Attention: blockwise attention on local KV).
 *   o_partial:   device fp32 [T_r,H,D], rows in rank-local order
 *                (index_map[rank_offsets[q_rank] + i] is the global row of i).
 *   lse_partial: device fp32 [H,T_r].
 *   Rows with no allowed key in the block get O = 0 and lse = -inf.
 * Merge the cp partials of a rank with cpattn_merge. */
cpattn_status_t cpattn_block_fwd(const cpattn_plan_t* plan, const void* q, const void* k,
                                 const void* v, cpattn_dtype_t dtype, int32_t H, int32_t Hkv,
                                 int32_t D, float scale, int32_t causal, int32_t q_rank,
                                 int32_t ring_step, float* o_partial, float* lse_partial,
                                 void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- backward
 *
 * Gradients of the packed attention for an upstream gradient dO, computed the
 * way blockwise ring attention trains ("Scaling video training with
 * parallelism", section 2, Ring Attention): the KV shard of virtual rank k
 * visits the query shards of ranks (k + t) mod cp at ring steps t = 0..cp-1,
 * collecting dK and dV, while each query shard collects dQ.  Softmax
 * probabilities are recomputed from the saved LSE:
 *   P = exp(scale q.k - lse), delta = rowsum(dO * O),
 *   dV = P^T dO,  dS = P * (dO V^T - delta),  dK = scale dS^T Q,  dQ = scale dS K
 * (dK and dV of a KV head sum over the query heads that read it).
 *   Supported: bf16 with D = 128 (tensor cores), fp32 with D = 64 or 128.
 *   Other shapes: CPATTN_UNSUPPORTED.
 *
 * Workspace bytes for cpattn_bwd / cpattn_block_bwd with this plan and shape
 * (work list, per-row scratch, a fp32 dQ accumulator [T,H,D], GRID2D shards). */
cpattn_status_t cpattn_bwd_workspace_size(const cpattn_plan_t* plan, int32_t H, int32_t Hkv, int32_t D,
                                          cpattn_dtype_t dtype, int32_t causal, size_t* bytes);

/* The whole packed backward.
 *   q, k, v, dout: device, the layouts of cpattn_fwd (dout like o);
 *   o, lse: the forward's outputs for these inputs (cpattn_fwd).
 *   dq [T,H,D], dk and dv [T,Hkv,D]: device outputs in the input dtype, every
 *   row written.  Reads no output before writing it.
 *   Errors as cpattn_fwd; CPATTN_WORKSPACE below cpattn_bwd_workspace_size. */
cpattn_status_t cpattn_bwd(const cpattn_plan_t* plan, const void* q, const void* k, const void* v,
                           const void* o, const float* lse, const void* dout, cpattn_dtype_t dtype,
                           int32_t H, int32_t Hkv, int32_t D, float scale, int32_t causal, void* dq,
                           void* dk, void* dv, void* workspace, size_t ws_bytes, void* stream);

/* One ring step of the backward: the gradients that rank `q_rank`'s queries
 * send through the KV shard of rank (q_rank - ring_step) mod cp, ADDED to
 * fp32 accumulators at global rows:
 *   dq_acc [T,H,D] += the step's dQ of rank q_rank's rows;
 *   dk_acc, dv_acc [T,Hkv,D] += the step's dK, dV of the KV shard's rows.
 * o and lse are the final (merged) forward outputs.  The cp steps of every
 * rank add up to the gradients of cpattn_bwd (up to rounding).  Steps must not
 * run concurrently on the same accumulators. */
cpattn_status_t cpattn_block_bwd(const cpattn_plan_t* plan, const void* q, const void* k, const void* v,
                                 const void* o, const float* lse, const void* dout, cpattn_dtype_t dtype,
                                 int32_t H, int32_t Hkv, int32_t D, float scale, int32_t causal,
                                 int32_t q_rank, int32_t ring_step, float* dq_acc, float* dk_acc,
                                 float* dv_acc, void* workspace, size_t ws_bytes, void* stream);

/* Exact log-sum-exp merge of n partials of the same rows:
 *   M = max_p lse_p;  lse = M + ln sum_p exp(lse_p - M);
 *   O = sum_p exp(lse_p - lse) * O_p.
 * Partials with lse = -inf contribute nothing; if all are -inf, O = 0 and
 * lse = -inf.  (The pages name blockwise ring attention but not its merge;
 * this is the identity that recombines softmax partials exactly.)
 *   o_parts_host / lse_parts_host: host arrays of n_partials (1..64) device
 *     pointers to fp32 [rows,H,D] and fp32 [H,rows].
 *   out_rows: device int64 [rows] giving the output row of each input row,
 *     or NULL for the identity; out_total_rows is the row count of o_out and
 *     the leading dimension of lse_out ([H,out_total_rows]).
 *   o_out: device [out_total_rows,H,D] of out_dtype; lse_out: device fp32. */
cpattn_status_t cpattn_merge(int32_t n_partials, const float* const* o_parts_host,
                             const float* const* lse_parts_host, int64_t rows, int32_t H,
                             int32_t D, const int64_t* out_rows, int64_t out_total_rows,
                             void* o_out, cpattn_dtype_t out_dtype, float* lse_out, void* stream);

/* Row permutation between global THD order and rank shards (the local
 * equivalents of split_cp_2d and gather_cp_2d, LongCat-Video article,
 * communication primitives).  `index` is device int64 [rows]:
 *   gather:  dst[i] = src[index[i]]   (global -> shard order); src has src_rows rows
 *   scatter: dst[index[i]] = src[i]   (shard -> global order); dst has dst_rows rows
 * A row whose index lies outside [0, src_rows) / [0, dst_rows) is skipped.
 * Each row is row_bytes bytes (a multiple of 16); buffers are 16-byte
 * aligned and must not overlap. */
cpattn_status_t cpattn_gather_rows(const void* src, int64_t src_rows, void* dst, const int64_t* index,
                                   int64_t rows, int64_t row_bytes, void* stream);
cpattn_status_t cpattn_scatter_rows(const void* src, void* dst, int64_t dst_rows, const int64_t* index,
                                    int64_t rows, int64_t row_bytes, void* stream);

/* Copy `bytes` from src to dst with a kernel, so that either side can be
 * pinned host memory that the GPU reads or writes directly over the host link
 * (NVLink-C2C on Grace hosts) instead of through a copy engine.  The pages
 * have no counterpart: this serves the end-to-end path that brings each
 * step's inputs from the host.
 *   dst, src: device memory or pinned (registered) host memory, 16-byte
 *     aligned, not overlapping; bytes a multiple of 16.
 *   n_blocks: thread blocks of 256 threads (<= 0: four per SM); fewer blocks
 *     leave room on the SMs for kernels running beside the copy.
 *   Errors: CPATTN_INVALID_ARG for NULL, misaligned or pageable pointers. */
cpattn_status_t cpattn_copy(void* dst, const void* src, size_t bytes, int32_t n_blocks, void* stream);

/* Bytes of device scratch compiled into the library for cpattn_fwd_static. */
#define CPATTN_STATIC_SCRATCH_BYTES (8u << 20)

/* The packed forward of cpattn_fwd for callers that cannot allocate device
 * memory: a plugin or operator interface that passes only input and output
 * buffers, or a process whose device memory belongs entirely to another
 * allocator.  (The pages have no counterpart: this is an interface
 * convenience, not a step of the method.)
 *   Same arguments and results as cpattn_fwd, without the workspace.  The
 *   call allocates no device or pinned host memory: its scratch (fault word
 *   and work list) is a fixed array of CPATTN_STATIC_SCRATCH_BYTES (8 MiB)
 *   inside the library, held on every GPU that loads the library until the
 *   process exits.
 *   The first call on each device finds the array's device address with
 *   cudaGetSymbolAddress (that device must be current); make that first call
 *   before any stream capture.
 *   Every call shares the one array and it keeps the last call's contents
 *   (each call clears the fault word and rewrites the work list), so calls
 *   that overlap on the GPU - on different streams, or from different
 *   threads - race: serialise them.
 *   The work list is copied from pageable host memory, so the call waits for
 *   work already queued on `stream` before it returns.
 *   Errors: CPATTN_WORKSPACE when the plan's work list does not fit in the
 *   array (the message gives both sizes); CPATTN_UNSUPPORTED for GRID2D,
 *   ULYSSES2D and PAIRED plans, whose shard gathers and all-to-all buffers
 *   need more scratch than the array holds.  A bounded wait that runs out
 *   inside the kernel records a fault in the array's header (the output is
 *   then incomplete); cpattn_static_sync_status reports it. */
cpattn_status_t cpattn_fwd_static(const cpattn_plan_t* plan, const void* q, const void* k, const void* v,
                                  cpattn_dtype_t dtype, int32_t H, int32_t Hkv, int32_t D, float scale,
                                  int32_t causal, void* o, float* lse, void* stream);

/* Synchronise `stream`, then report a fault that a cpattn_fwd_static kernel
 * recorded in the static array of the current device (CPATTN_DEVICE_FAULT,
 * with the block and the wait in the message) or a CUDA error
 * (CPATTN_CUDA_ERROR).  Allocates nothing: the header is copied by symbol
 * into host stack memory.  The next cpattn_fwd_static call on the device
 * clears the fault word.  Like the array, the word is shared by every call:
 * check it before the next call is issued. */
cpattn_status_t cpattn_static_sync_status(void* stream);

/* --------------------------------------------------------------- loss, FLOPs */

/* Per-token loss normalisation over valid tokens (Dynamic-CP article, section
 * "Loss computation and FLOPS statistics"):
 *   *out_loss = sum_t [valid_t != 0] loss_t / sum_t [valid_t != 0]
 * accumulated in fp64 in a fixed order (deterministic), *out_count the exact
 * number of valid tokens.  With no valid token *out_loss = 0.
 *   loss: device fp32 [T]; valid: device uint8 [T] (0 = padding).
 *   out_loss: device fp64 scalar; out_count: device int64 scalar;
 *   out_loss_f32: device fp32 scalar or NULL. */
cpattn_status_t cpattn_token_loss_norm(const float* loss, const uint8_t* valid, int64_t T,
                                       double* out_loss, int64_t* out_count, float* out_loss_f32,
                                       void* stream);

/* THD-aware forward FLOPs, 4*D*H*sum_s pairs(L_s), pairs = L(L+1)/2 causal,
 * L^2 otherwise; counted from the real lengths, never max_seqlen (Dynamic-CP
 * article, section "Loss computation and FLOPS statistics").  Exact integer
 * in *out_u64 (may be NULL), the same as a double in *out_f64 (may be NULL). */
cpattn_status_t cpattn_fwd_flops(const int32_t* cu_seqlens_host, int32_t n_seqs, int32_t H,
                                 int32_t D, int32_t causal, uint64_t* out_u64, double* out_f64);

/* ------------------------------------------------- Dynamic-CP scheduler (host)
 *
 * Per-micro-batch CP size and packing of a global batch of variable-length
 * samples ("Speeding up Variable-Length Training with Dynamic Context
 * Parallelism and NVIDIA Megatron Core", data-scheduling section, Eq. 1-3, and
 * the runtime section's grid search over the micro-batch count).  Host
 * functions: no device memory, no stream.  A micro-batch's samples, packed in
 * ascending sample order, give the cu_seqlens and its CP size the cp_size of
 * cpattn_plan.
 *
 * Workload model: workload(S) = attn_coef * S(S+1)/2 + lin_coef * S (the
 * O(S^2) attention and O(S) per-token parts; attn_coef = 4*D*H makes the first
 * term the causal attention FLOP count); memory(S) = S tokens.
 * Readings of the prose: every micro-batch has the quota
 * Q = ceil(total / n_micro); a sample's CP size is the smallest power of two
 * c <= max_cp with workload <= c*Q and S <= c*cap_tokens (else max_cp); the
 * n_micro lowest-workload samples open one micro-batch each; every other
 * sample, by descending workload, joins the micro-batch with the least
 * per-GPU load after the placement, load = workload * (max_cp / cp), among
 * those whose tokens stay <= cp * cap_tokens, else the least-loaded one; a
 * micro-batch's CP size is the largest of its samples'; ties go to the lower
 * index.  Integer arithmetic throughout: results are exact and deterministic. */
typedef struct cpattn_dcp_config {
  int32_t max_cp;      /* largest CP group, a power of two in [1, 1024] */
  int32_t reserved;    /* 0 */
  int64_t cap_tokens;  /* activation memory cap: tokens one GPU holds (>= 1) */
  int64_t attn_coef;   /* workload units per causal (query, key) pair (>= 0) */
  int64_t lin_coef;    /* workload units per token (>= 0) */
} cpattn_dcp_config_t;

/* Eq. 1-3: per-micro-batch workload W_i of DP rank i with m[i] micro-batches,
 * V = vpp virtual stages and p = pp pipeline stages, such that
 * W_i (m_i V + p - 1) is the same on every rank and sum_i W_i m_i = total.
 *   m: host int32 [dp] (each >= 1); w_out: host fp64 [dp].
 *   Errors: CPATTN_INVALID_ARG for dp, vpp or pp < 1, m[i] < 1, or a negative
 *   or non-finite total. */
cpattn_status_t cpattn_dcp_quotas(const int32_t* m, int32_t dp, int32_t vpp, int32_t pp, double total,
                                  double* w_out);

/* Packs n samples into n_micro micro-batches and picks their CP sizes.
 *   seqlens: host int64 [n], each in [1, 2^40].  Outputs (host, any may be
 *   NULL): sample_micro [n] and sample_cp [n]; micro_cp, micro_work,
 *   micro_tokens [n_micro] (a micro-batch with no sample has cp 1, work 0).
 *   Errors: CPATTN_INVALID_ARG for a bad config, n_micro < 1, a length out of
 *   range, or total workload * max_cp beyond int64. */
cpattn_status_t cpattn_dcp_schedule(const int64_t* seqlens, int64_t n, const cpattn_dcp_config_t* cfg,
                                    int32_t n_micro, int32_t* sample_micro, int32_t* sample_cp,
                                    int32_t* micro_cp, int64_t* micro_work, int64_t* micro_tokens);

/* Grid search over the micro-batch count m per DP rank (the same on every
 * rank), m = pp .. mult*pp: budgets[m - pp] = the largest per-GPU load
 * (workload * max_cp / cp) of cpattn_dcp_schedule with dp*m micro-batches.
 * *knee_m = the knee of that curve: the m farthest below the chord from its
 * first to its last point with both axes scaled to [0, 1] (the first m when
 * the curve does not fall).  *best_m = the m in {knee-1, knee, knee+1} with
 * the least Eq. 1 step time budget * (m*vpp + pp - 1) (the reading used in
 * place of the pages' pipeline simulator).  Ties go to the smaller m.
 *   budgets: host int64 [(mult-1)*pp + 1] or NULL; knee_m, best_m may be NULL.
 *   Errors: CPATTN_INVALID_ARG as cpattn_dcp_schedule, or dp, pp, vpp,
 *   mult < 1, or dp*mult*pp > 2^20. */
cpattn_status_t cpattn_dcp_sweep(const int64_t* seqlens, int64_t n, const cpattn_dcp_config_t* cfg, int32_t dp,
                                 int32_t pp, int32_t vpp, int32_t mult, int64_t* budgets, int32_t* knee_m,
                                 int32_t* best_m);

/* ----------------------------------------------------------------- helpers */

/* Synchronise `stream`, then report a fault recorded by a kernel in
 * `workspace` (CPATTN_DEVICE_FAULT) or a CUDA error (CPATTN_CUDA_ERROR).
 * The fault word is cleared by the next cpattn_fwd / cpattn_block_fwd. */
cpattn_status_t cpattn_sync_status(const void* workspace, void* stream);

/* Test support for the device fault path (not for production use).
 * Process-wide settings applied to the workspace of every later cpattn_fwd,
 * cpattn_block_fwd, cpattn_bwd and cpattn_block_bwd call:
 *   wait_limit_us: every bounded wait inside the kernels gives up after this
 *     many microseconds instead of the default 4 s (0 restores the default);
 *   withhold_first_v: nonzero makes block 0 of the bf16 forward skip loading
 *     its first V tile, so the MMA thread's wait for it (and the waits of the
 *     warps behind it) run out: the kernel records a wait timeout (fault code
 *     1, block 0, the site that ran out first) in the workspace, lets
 *     its copies in flight land, frees its tensor memory and returns early;
 *     the output is then incomplete and cpattn_sync_status reports
 *     CPATTN_DEVICE_FAULT.
 * No GPU fault, trap or hang is involved: only a wait that nothing completes,
 * ended by its time limit.  Errors: CPATTN_INVALID_ARG for withhold_first_v
 * without a limit, or a limit above 10 s. */
cpattn_status_t cpattn_debug_wait_fault(uint32_t wait_limit_us, int32_t withhold_first_v);

/* Message of the last failed call on this thread ("" if none). */
const char* cpattn_last_error_string(void);

/* Library version string. */
const char* cpattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CPATTN_H */
