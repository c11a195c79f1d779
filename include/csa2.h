/*
 * csa2.h - C ABI of the CSA2 attention step (DeepSeek-V4.1-Flash) on sm_103a.
 *
 * The step, as the pages describe it ("DeepSeek-V4.1-Flash explained", sections 2 and 3;
 * "Every layer, connected", "The global and index paths" and "The query and output
 * paths"; "DeepSeek V4 Inside", CSA section and eq. (27)):
 *
 *   1. the lightning indexer scores every causally visible global record,
 *        score_j = sum_{h<32} w_h * ReLU(q^I_h . k^I_j);
 *   2. top-K (512) selection of record addresses, directly or from a block-max pool
 *      built by the first decoder indexer (hierarchical indexing); Reuse layers take
 *      the preceding layer's selection;
 *   3. 64-head x 512 shared-latent MQA over the selected latents (each latent is key and
 *      value at once) plus the layer's 128-token sliding window, one sink logit per head
 *      in the softmax denominator, RoPE on the last 64 dims of q and inverse RoPE on the
 *      output's rotary coordinates.
 *
 * Around the step (the calls after csa2_fused_decode below): the cache writer (records
 * rotated and stored as FP4, FP8 or bf16 rows), the encoder's sequence compressor, the
 * expansion of MXFP4 indexer keys for prefill, a plain projection (csa2_linear), and the
 * query low-rank path and grouped output projection on either side of attention.
 *
 * Conventions shared by every call
 *   - Every pointer in an args struct is a DEVICE pointer owned by the caller, unless a
 *     field says otherwise.  The library keeps no pointer after the call returns.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL = the
 *     legacy default stream).  They never synchronize and never allocate; scratch memory
 *     comes from the caller through `workspace` (size from the matching *_workspace_size).
 *     One call is the exception: csa2_read_device_status copies a status word to the host
 *     and therefore synchronizes its stream.
 *   - Arrays are dense row-major; base pointers must be 16-byte aligned.
 *   - Arguments are validated on the host before anything is launched.  An invalid call
 *     returns CSA2_EINVAL (or CSA2_EUNSUPPORTED for a valid request outside the
 *     implemented sizes) and launches nothing.  CSA2_ECUDA reports a failed launch.
 *   - Device pointer contents are not inspected by the host.  Attention skips a selected
 *     record index outside [0, n_records) (other than the -1 pad) and, when `dev_status` is
 *     given, stores CSA2_EDEVICE_INDEX there.  Other out-of-range device data (a sequence
 *     index >= n_seq, a candidate position >= n_records, n_visible > n_records) is
 *     undefined behaviour.
 *   - Fixed sizes: 32 indexer heads x 128 dims; 64 query heads x 512 dims; RoPE on the
 *     last 64 dims (adjacent pairs, frequency theta^(-2i/64)).
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CSA2_IDX_HEADS 32
#define CSA2_IDX_DIM 128
#define CSA2_HEADS 64
#define CSA2_HEAD_DIM 512
#define CSA2_ROPE_DIM 64
#define CSA2_MAX_TOPK 1024

typedef enum csa2_status {
  CSA2_OK = 0,
  CSA2_EINVAL = 1,          /* bad shape, dtype, null pointer or alignment; nothing launched */
  CSA2_EUNSUPPORTED = 2,    /* a valid request outside the implemented sizes */
  CSA2_ECUDA = 3,           /* a CUDA launch or runtime call failed */
  CSA2_ETIMEOUT = 4,        /* a device-side bounded wait gave up (reported in dev_status) */
  CSA2_EWORKSPACE = 5,      /* workspace missing or smaller than *_workspace_size */
  CSA2_EDEVICE_INDEX = 6    /* a kernel met (and skipped) an out-of-range device index */
} csa2_status;

/* Storage formats of cached rows. */
typedef enum csa2_dtype {
  CSA2_BF16 = 0,              /* bf16 values */
  CSA2_FP8_E4M3_ROWSCALE = 1, /* OCP E4M3 codes, one fp32 scale per row: value = code * scale */
  CSA2_FP4_E2M1_G32 = 2,      /* E2M1 codes, two per byte (low nibble = even channel), and one
                                 E4M3 scale per 32 channels in a separate array:
                                 value = level * scale ("DeepSeek-V4.1-Flash explained", section 7) */
  CSA2_FP4_E2M1_G16 = 3,      /* the same with one scale per 16 channels, as the pages state */
  CSA2_MXFP4 = 4              /* indexer keys only: OCP MXFP4, E2M1 codes two per byte (low nibble
                                 = even element) and one UE8M0 exponent per block of 32 in
                                 k_scale [n_seq, n_records, 4] uint8: value = level * 2^(e-127)
                                 (the pages' indexer precision, "DeepSeek-V4.1-Flash explained",
                                 section 7) */
} csa2_dtype;

/* Layer modes of a CSA2 sharing group ("DeepSeek-V4.1-Flash explained", section 2, mode
 * table; section 3 for the pool). */
typedef enum csa2_mode {
  CSA2_MODE_FULL = 0,       /* score all visible records, fresh top-K, attend */
  CSA2_MODE_FULL_POOL = 1,  /* FULL, and also build the block pool for later indexers */
  CSA2_MODE_REINDEX = 2,    /* score only the pool with this layer's indexer query, top-K, attend */
  CSA2_MODE_REUSE = 3       /* no indexing: attend over the given selection */
} csa2_mode;

/* ------------------------------------------------------------------------------------
 * csa2_index_scores - lightning-indexer scores.
 *
 * The indexer adds up the rectified query-key dot products of 32 heads, each with its own
 * weight, and only causally visible records may be selected ("Every layer, connected",
 * "The global and index paths").
 *   scores[r, j] = sum_h w[r, h] * max(0, q_idx[r, h, :] . key(j))       for a candidate j
 *   scores[r, j] = -inf                                                   otherwise
 * One indexer key per record, shared by all 32 heads.  FP8 keys: key(j) = code * k_scale[j].
 * MXFP4 keys (k_dtype CSA2_MXFP4, k_idx [n_seq, n_records, 64] uint8, k_scale the exponents
 * [n_seq, n_records, 4] uint8): key(j)[d] = level(d) * 2^(e(j, d / 32) - 127).  MXFP4
 * indexer queries are given as their (exact) bf16 values.
 * Without `cand`, j runs over records 0..n_records-1 and records >= n_visible[r] are not
 * candidates.  With `cand`, j runs over cand[r, 0..L) (record positions, strictly
 * ascending, e.g. a block pool) and entries >= n_cand[r] are not candidates.
 * Optionally also the block maxima: block_max[r, c] = max over the candidate records of
 * block c = [c*block_size, (c+1)*block_size) (-inf if none), for the block pool.
 * ------------------------------------------------------------------------------------ */
typedef struct csa2_index_args {
  const void* q_idx;          /* [n_rows, 32, 128] bf16 */
  const float* w;             /* [n_rows, 32] */
  const void* k_idx;          /* [n_seq, n_records, 128]: bf16, or E4M3 bytes (k_dtype FP8) */
  const float* k_scale;       /* [n_seq, n_records] row scales for FP8 keys; MXFP4: the exponent
                                 bytes [n_seq, n_records, 4] (passed through this pointer); else NULL */
  int32_t k_dtype;            /* CSA2_BF16, CSA2_FP8_E4M3_ROWSCALE or CSA2_MXFP4 */
  int32_t n_rows;             /* query rows (>= 0) */
  int32_t n_seq;              /* sequences sharing the key layout */
  int64_t n_records;          /* records per sequence (>= 1) */
  const int32_t* seq_of_row;  /* [n_rows] sequence of each query row */
  const int32_t* n_visible;   /* [n_rows] records 0..n_visible-1 are visible (<= n_records) */
  const int32_t* cand;        /* [n_rows, L] candidate record positions, or NULL */
  const int32_t* n_cand;      /* [n_rows] valid candidates per row (required with cand) */
  int64_t L;                  /* candidates per row when cand != NULL */
  float* scores;              /* out [n_rows, L or n_records] fp32 */
  float* block_max;           /* out [n_rows, ceil(n_records / block_size)] or NULL (no cand) */
  int32_t block_size;         /* > 0 when block_max != NULL */
} csa2_index_args;

csa2_status csa2_index_scores(const csa2_index_args* a, void* stream);

/* ------------------------------------------------------------------------------------
 * csa2_topk - exact top-K of every row, returned as addresses.
 *
 * Selection yields record addresses, not scores, and equal scores go to the lower
 * position (course lesson "06 / Indexer and attention", select_values).  Entries 0..n_valid[r]-1 of row r are the
 * candidates; the K best by (score descending, entry index ascending) are selected, with
 * -0.0 == +0.0.  idx[r] holds their record positions (cand[r, j], or j when cand is NULL)
 * as an ASCENDING set, padded with -1 when fewer than K are valid.  Scores must not be NaN.
 * ------------------------------------------------------------------------------------ */
typedef struct csa2_topk_args {
  const float* scores;        /* [n_rows, L] */
  const int32_t* cand;        /* [n_rows, L] strictly ascending record positions, or NULL */
  const int32_t* n_valid;     /* [n_rows] in [0, L] */
  int32_t n_rows;
  int64_t L;                  /* 1 .. 2^24 */
  int32_t K;                  /* 1 .. CSA2_MAX_TOPK */
  int32_t* idx;               /* out [n_rows, K] */
  void* workspace;            /* csa2_topk_workspace_size bytes */
  size_t workspace_bytes;
} csa2_topk_args;

size_t csa2_topk_workspace_size(const csa2_topk_args* a);
csa2_status csa2_topk(const csa2_topk_args* a, void* stream);

/* ------------------------------------------------------------------------------------
 * csa2_topk_static - csa2_topk without a caller-provided workspace.  (The pages describe no
 * counterpart: this is a library convenience, not part of the method.)
 *
 * For callers that cannot allocate device memory - a framework capturing the stream into a
 * CUDA graph while it owns every allocation, or a runtime with a fixed memory budget that
 * admits no allocation once it runs - the scratch memory of csa2_topk comes from a
 * device-global array inside the library, CSA2_TOPK_STATIC_SCRATCH_BYTES bytes that every
 * GPU loading the library holds until the process exits.  The call allocates nothing; the
 * caller passes inputs and outputs exactly as for csa2_topk (a->workspace is ignored).
 *   - Results are those of csa2_topk.
 *   - The scratch is 8 bytes per (row segment, K) pair plus 8 per row segment, and rows
 *     are split into at most one segment per multiprocessor in total, so on the supported
 *     GPU (152 multiprocessors) every valid request needs at most 1.3 MB and fits: the
 *     CSA2_EUNSUPPORTED answer for a request whose scratch would exceed the array is a
 *     guard that such a device never reaches.
 *   - `stream` must belong to the current device (the array and the segment count are
 *     those of the current device); a stream of another device returns CSA2_EINVAL.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 *     with that device current; make that first call before any stream capture.  The
 *     address is remembered for the life of the process: after cudaDeviceReset the library
 *     must not be used again on that device.
 *   - All calls on a device share the one array, which keeps the last call's contents
 *     (nothing in it needs to start at zero).  Calls that may overlap on the GPU - on
 *     different streams without ordering between them - race on it and must be serialised
 *     by the caller.
 * ------------------------------------------------------------------------------------ */
#define CSA2_TOPK_STATIC_SCRATCH_BYTES (2u << 20)
csa2_status csa2_topk_static(const csa2_topk_args* a, void* stream);

/* ------------------------------------------------------------------------------------
 * csa2_block_pool - the hierarchical candidate pool of the first decoder indexer.
 *
 * The first decoder indexer cuts the positions into blocks, rates each block by its best
 * position and keeps the best blocks; later Reindex layers select only among those
 * ("DeepSeek-V4.1-Flash explained", section 3; course lesson "07 / Hierarchical
 * indexing").  Of the ceil(n_visible[r] / block_size) blocks of row r, the n_keep best by
 * (block max descending, block index ascending) are kept; pool[r] lists every visible
 * position of the kept blocks in ascending order, -1 padded; n_pool[r] is its length.
 * ------------------------------------------------------------------------------------ */
typedef struct csa2_block_pool_args {
  const float* block_max;     /* [n_rows, n_blocks] from csa2_index_scores */
  const int32_t* n_visible;   /* [n_rows] */
  int32_t n_rows;
  int32_t n_blocks;           /* ceil(n_records / block_size) */
  int32_t block_size;         /* 1 .. 4096 */
  int32_t n_keep;             /* 1 .. n_keep * block_size <= 2^20 */
  int32_t* pool;              /* out [n_rows, n_keep * block_size] */
  int32_t* n_pool;            /* out [n_rows] */
  void* workspace;            /* csa2_block_pool_workspace_size bytes */
  size_t workspace_bytes;
} csa2_block_pool_args;

size_t csa2_block_pool_workspace_size(const csa2_block_pool_args* a);
csa2_status csa2_block_pool(const csa2_block_pool_args* a, void* stream);

/* ------------------------------------------------------------------------------------
 * csa2_sparse_attn - shared-latent MQA over the selected latents plus the sliding window.
 *
 * For query row r at position p = q_pos[r] of sequence b = seq_of_row[r]:
 *   q'_h  = RoPE_p(q[r, h])            on dims 448..511, pairs (448+2i, 449+2i), angle
 *                                      p * rope_theta^(-2i/64)
 *   rows  = latents[b, idx[r, k]] for idx != -1, then the window rows of positions
 *           max(p - window + 1, swa_pos0[b]) .. p (the current token included), read from
 *           swa[b, position - swa_pos0[b]]
 *   z_hj  = softmax_scale * q'_h . row_j
 *   o_h   = sum_j exp(z_hj) row_j / (sum_j exp(z_hj) + exp(sink[h]))    ("DeepSeek V4
 *           Inside", eq. (27): the sink logit is in the denominator only)
 *   out   = RoPE_{-p}(o_h) on dims 448..511 ("Every layer, connected", "The query and output
 *           paths": inverse RoPE on the output's rotary coordinates)
 *   sink_mass[r, h] = exp(sink[h]) / (sum_j exp(z_hj) + exp(sink[h]))
 * Latents and window rows are used as stored: the cache holds them already rotated.
 * Requires p - swa_pos0[b] < swa_rows.  FP8 window rows: row = code * swa_scale[row].
 * ------------------------------------------------------------------------------------ */
typedef struct csa2_attn_args {
  const void* q;              /* [n_rows, 64, 512] bf16, before RoPE */
  const int64_t* q_pos;       /* [n_rows] */
  const int32_t* seq_of_row;  /* [n_rows] */
  int32_t n_rows;
  int32_t n_seq;
  int64_t n_records;
  const void* latents;        /* bf16 [n_seq, n_records, 512] or FP4 codes [n_seq, n_records, 256] */
  const uint8_t* lat_scale;   /* FP4: E4M3 [n_seq, n_records, 512/group], else NULL */
  int32_t lat_dtype;          /* CSA2_BF16, CSA2_FP4_E2M1_G32 or CSA2_FP4_E2M1_G16 */
  const int32_t* idx;         /* [n_rows, K] record positions in [0, n_records) or -1 */
  int32_t K;                  /* 0 .. CSA2_MAX_TOPK */
  const void* swa;            /* bf16 [n_seq, swa_rows, 512] or E4M3 [n_seq, swa_rows, 512] */
  const float* swa_scale;     /* FP8: [n_seq, swa_rows], else NULL */
  int32_t swa_dtype;          /* CSA2_BF16 or CSA2_FP8_E4M3_ROWSCALE */
  int64_t swa_rows;
  const int64_t* swa_pos0;    /* [n_seq] absolute position of window row 0 */
  int32_t window;             /* 0 .. 1024 */
  const float* sink;          /* [64] sink logits */
  float rope_theta;           /* > 0 */
  float softmax_scale;
  void* out;                  /* out [n_rows, 64, 512] fp32 (bf16 with out_bf16) */
  float* sink_mass;           /* out [n_rows, 64] or NULL */
  void* workspace;            /* csa2_sparse_attn_workspace_size bytes: the partial results of
                                 each 128-entry tile (K + window entries per row) */
  size_t workspace_bytes;
  int32_t* dev_status;        /* optional device int32, set to CSA2_EDEVICE_INDEX when idx holds a
                                 record index outside [0, n_records) other than -1, or to
                                 CSA2_ETIMEOUT when a bounded wait on the tensor cores gave up
                                 (outputs then undefined); or NULL */
  int32_t out_bf16;           /* 0: out is fp32; 1: out is bf16 [n_rows, 64, 512] (each value the
                                 fp32 result rounded to nearest even), the input of
                                 csa2_out_proj */
} csa2_attn_args;

size_t csa2_sparse_attn_workspace_size(const csa2_attn_args* a);
csa2_status csa2_sparse_attn(const csa2_attn_args* a, void* stream);

/* ------------------------------------------------------------------------------------
 * csa2_fused_decode - one CSA2 layer of a decode step, with no host round trip.
 *
 * FULL:      index (all visible records) -> top-K -> attention.
 * FULL_POOL: FULL, and the block pool (block_size, n_keep) written to pool / n_pool.
 * REINDEX:   index over pool / n_pool (inputs) with this layer's q_idx and w -> top-K ->
 *            attention.
 * REUSE:     attention over idx (input).
 * Each layer has a fixed mode (course lesson "05 / Sharing memory"); a sharing group is a
 * sequence of calls on one stream.
 * The `index` member is read for FULL, FULL_POOL and REINDEX; its scores / block_max /
 * cand fields are ignored (the fused path keeps scores on chip).  The `attn` member's idx
 * field is ignored: attention reads `idx` below.
 * ------------------------------------------------------------------------------------ */
typedef struct csa2_decode_args {
  int32_t mode;               /* csa2_mode */
  csa2_index_args index;
  int32_t K;                  /* top-K (1 .. CSA2_MAX_TOPK) */
  int32_t block_size;         /* FULL_POOL */
  int32_t n_keep;             /* FULL_POOL */
  int32_t pool_len;           /* columns of pool: n_keep * block_size */
  int32_t* pool;              /* FULL_POOL: out; REINDEX: in  [n_rows, pool_len] */
  int32_t* n_pool;            /* FULL_POOL: out; REINDEX: in  [n_rows] */
  int32_t* idx;               /* FULL, FULL_POOL, REINDEX: out; REUSE: in  [n_rows, K] */
  csa2_attn_args attn;
  void* workspace;            /* csa2_fused_decode_workspace_size bytes, any contents (the
                                 per-row completion counters it holds carry a per-call tag,
                                 so nothing needs clearing between calls) */
  size_t workspace_bytes;
  /* Optional tracing: cudaEvent_t handles (as void*) recorded on `stream` at the stage
   * boundaries: [0] right before the indexer scan kernel (after the reset of its row
   * counters), [1] after it, [2] after the top-K merge and block pool (if any), [3] after
   * attention.  NULL entries are skipped.  Each record adds a short gap between the
   * kernels.  The events belong to the caller, who must have created them (cudaEventCreate). */
  void* stage_events[4];
} csa2_decode_args;

size_t csa2_fused_decode_workspace_size(const csa2_decode_args* a);
/* Number of kernels one csa2_fused_decode call with these arguments launches. */
int32_t csa2_fused_decode_launch_count(const csa2_decode_args* a);
csa2_status csa2_fused_decode(const csa2_decode_args* a, void* stream);

/* ------------------------------------------------------------------------------------
 * Splitting one sequence's records across devices.  A long context's records can be cut into
 * contiguous ranges, one per device: every record's score needs only that record's key, and
 * the row's top-K is a subset of the union of every range's own top-K, so each device
 *   1. scores its range (csa2_index_scores with the range's keys, n_records = the range's
 *      length and n_visible = the row's visible records inside the range),
 *   2. keeps the range's exact top-K as a candidate list (csa2_shard_candidates),
 * the lists of all ranges are gathered (all ranges' lists, in range order, on every device),
 *   3. every device merges them into the row's top-K (csa2_merge_candidates: the same answer
 *      on every device, bit for bit),
 *   4. attends over the selected records of its own range (its indices, the others -1) and,
 *      on the device that holds them, the window rows, into partials
 *      (csa2_sparse_attn_partial: per 128-entry tile and head the maximum logit, the sum of
 *      exp(logit - maximum) and the output relative to it),
 * the partials are gathered, and
 *   5. csa2_attn_merge combines them: log-sum-exp over every part's tiles, the sink in the
 *      denominator, normalisation and the inverse rotation ("DeepSeek V4 Inside", eq. (27)).
 * The result equals csa2_fused_decode's FULL layer on the whole sequence (indices bit-exact).
 * On one device the ranges simply run one after another.
 * ------------------------------------------------------------------------------------ */
typedef struct csa2_shard_args {
  const float* scores;        /* [n_rows, L] the range's indexer scores */
  const int32_t* n_valid;     /* [n_rows] visible records of the range (its columns 0 .. n_valid-1) */
  int32_t n_rows;
  int64_t L;                  /* records in the range, 1 .. 2^24 */
  int32_t K;                  /* 1 .. CSA2_MAX_TOPK */
  int64_t first_record;       /* record position of column 0 (>= 0) */
  float* out_scores;          /* out [n_rows, K] the selected entries' scores in ascending position
                                 order, -inf after them */
  int32_t* out_pos;           /* out [n_rows, K] their record positions (first_record + column), -1
                                 after them */
  int32_t* out_cnt;           /* out [n_rows] entries listed: min(K, n_valid) */
  void* workspace;            /* csa2_shard_candidates_workspace_size bytes */
  size_t workspace_bytes;
} csa2_shard_args;

size_t csa2_shard_candidates_workspace_size(const csa2_shard_args* a);
csa2_status csa2_shard_candidates(const csa2_shard_args* a, void* stream);

/* The row's top-K of n_lists candidate lists (the K best by score descending, position
 * ascending, of every list's first cnt entries), returned as the ascending set of positions,
 * -1 padded.  The lists come as gathered, list-major (list l = range l's csa2_shard_candidates
 * output), in ascending position ranges (each list ascending). */
typedef struct csa2_merge_args {
  const float* scores;        /* [n_lists, n_rows, K_in] */
  const int32_t* pos;         /* [n_lists, n_rows, K_in] */
  const int32_t* cnt;         /* [n_lists, n_rows] entries of each list, 0 .. K_in */
  int32_t n_rows;
  int32_t n_lists;            /* 1 .. 64 */
  int32_t K_in;               /* 1 .. CSA2_MAX_TOPK */
  int32_t K;                  /* 1 .. CSA2_MAX_TOPK */
  int32_t* idx;               /* out [n_rows, K] */
  void* workspace;            /* csa2_merge_candidates_workspace_size bytes, 16-byte aligned */
  size_t workspace_bytes;
} csa2_merge_args;

size_t csa2_merge_candidates_workspace_size(const csa2_merge_args* a);
csa2_status csa2_merge_candidates(const csa2_merge_args* a, void* stream);

/* Attention partials of one device's share: csa2_sparse_attn's arguments (attn.out, sink_mass,
 * sink and workspace are not used) with attn.idx holding the selected records of this
 * device's range (-1 elsewhere) and attn.window the window rows it holds (0 for none).
 * Writes, per row, 128-entry tile t (entries K + window in tiles, csa2_attn_partial_tiles) and
 * head h: part_ml[row, t, h] = (maximum logit m, sum of exp(logit - m)) and
 * part_o[row, t, h, :] = sum of exp(logit - m) * row, before the inverse rotation. */
typedef struct csa2_partial_args {
  csa2_attn_args attn;
  float* part_o;              /* out [n_rows, tiles, 64, 512], 16-byte aligned */
  float* part_ml;             /* out [n_rows, tiles, 64, 2] */
  int64_t range_first;        /* with range_count > 0: attn.idx holds global positions (the merged
                                 selection); those outside [range_first, range_first + range_count)
                                 are skipped and the others read attn.latents at position -
                                 range_first (this device's records only); range_count == 0: attn.idx
                                 indexes attn.latents directly */
  int64_t range_count;
  int32_t skip_window;        /* 1: the window entries are masked (another device attends to them);
                                 the tiles stay csa2_attn_partial_tiles(K, window) */
} csa2_partial_args;

int32_t csa2_attn_partial_tiles(int32_t K, int32_t window);
csa2_status csa2_sparse_attn_partial(const csa2_partial_args* a, void* stream);

/* The output of n_parts gathered partials (part k = one device's part_o / part_ml, stacked):
 * o_h = sum over every tile of exp(m - M) o_tile / (sum exp(m - M) l_tile + exp(sink[h] - M)),
 * then turned back by -q_pos on dims 448..511; sink_mass as csa2_sparse_attn's. */
typedef struct csa2_attn_merge_args {
  const float* part_o;        /* [n_parts, n_rows, part_tiles, 64, 512] */
  const float* part_ml;       /* [n_parts, n_rows, part_tiles, 64, 2] */
  int32_t n_parts;
  int32_t part_tiles;         /* n_parts * part_tiles <= 32 */
  int32_t n_rows;
  const int64_t* q_pos;       /* [n_rows] */
  const float* sink;          /* [64] */
  float rope_theta;
  void* out;                  /* out [n_rows, 64, 512] fp32, or bf16 with out_bf16 */
  int32_t out_bf16;
  float* sink_mass;           /* out [n_rows, 64] or NULL */
} csa2_attn_merge_args;

csa2_status csa2_attn_merge(const csa2_attn_merge_args* a, void* stream);

/* ------------------------------------------------------------------------------------
 * Cache writer: appends records to a main-KV (latent) cache or a sliding-window cache in its
 * storage format.  Each record's rotary coordinates (dims 448..511, pairs (448+2i, 449+2i),
 * frequencies theta^(-2i/64)) are turned by its position first, since the cache holds
 * rotated values and is quantized after RoPE (course, FP4 lesson, section 4, "Quantize after
 * RoPE"); then:
 *   FP4 (CSA2_FP4_E2M1_G16 / _G32): per group of 16 / 32 channels the E4M3 scale is the
 *     smallest E4M3 value >= amax / 6 (so no element clips; saturating at 448), and each
 *     value / scale rounds to the nearest E2M1 level, ties to the even code; codes two per
 *     byte, low nibble = even channel ("DeepSeek-V4.1-Flash explained", section 7: one E4M3
 *     scale per 16 channels; the scale selection itself is not described by the pages);
 *   FP8 (CSA2_FP8_E4M3_ROWSCALE): one fp32 scale amax / 448 per row (1 for an all-zero row),
 *     codes = E4M3(value / scale), round to nearest even (the local cache stays FP8, same
 *     lesson, section 4).
 * Every decision (divisions, the rotation's products and sums) is taken in IEEE float32; the
 * rotation's cos and sin are computed in double and rounded to float.
 * ------------------------------------------------------------------------------------ */
typedef struct {
  int64_t n_rows;             /* records to write */
  const void* x;              /* [n_rows, 512] values before rotation: float32 (x_f32 = 1) or bf16 */
  int32_t x_f32;
  const int64_t* pos;         /* [n_rows] position of each record, or NULL: no rotation */
  float rope_theta;
  const int64_t* dst_row;     /* [n_rows] row of the cache written (sequence * N + position for a
                                 [seq, N, ...] cache); rows outside [0, cache_rows) are skipped
                                 and reported through dev_status */
  int64_t cache_rows;
  int32_t out_dtype;          /* CSA2_FP4_E2M1_G16, CSA2_FP4_E2M1_G32, CSA2_FP8_E4M3_ROWSCALE or
                                 CSA2_BF16 (the rotated record rounded to nearest even) */
  void* codes;                /* [cache_rows, 256] (FP4) or [cache_rows, 512] (FP8) uint8, or
                                 [cache_rows, 512] bf16 */
  void* scales;               /* FP4: [cache_rows, 512 / G] E4M3 uint8; FP8: [cache_rows] float32;
                                 bf16: unused (may be NULL) */
  int32_t* dev_status;        /* optional device int32: CSA2_EDEVICE_INDEX on a skipped row */
} csa2_write_args;

/* All pointers device, 16-byte aligned (pos, dst_row and FP8 scales: 8 / 8 / 4).  Rows are
 * written in any order; two records with the same dst_row leave either one. */
csa2_status csa2_write_records(const csa2_write_args* a, void* stream);

/* ------------------------------------------------------------------------------------
 * Sequence compressor of the encoder's global banks: entry e pools the `ratio` consecutive
 * tokens ratio*e .. ratio*e + ratio - 1 with channel-wise softmax gates,
 *   entry[e, c] = sum_j softmax_j(gate[ratio*e + j, c]) * kv[ratio*e + j, c]
 * (course, "How CSA2 compresses, shares, and selects attention memory": learned,
 * channel-wise softmax gates above ratio 1, no pooling at ratio 1; the encoder's banks use
 * ratio 2).  kv and gate are the tokens' projections (their weights are outside this call).
 * An entry is visible to a query at position p when all its tokens are: the first
 * (p + 1) / ratio entries, to be passed as n_visible to the indexer and attention calls.
 * ------------------------------------------------------------------------------------ */
typedef struct {
  int64_t n_entries;          /* entries formed */
  int32_t ratio;              /* 1 .. 8 */
  const void* kv;             /* [n_entries * ratio, 512] float32 (x_f32 = 1) or bf16 */
  const void* gate;           /* [n_entries * ratio, 512], the same type */
  int32_t x_f32;
  float* out;                 /* [n_entries, 512] float32 */
} csa2_compress_args;

/* All pointers device, 16-byte aligned. */
csa2_status csa2_compress(const csa2_compress_args* a, void* stream);

/* ------------------------------------------------------------------------------------
 * Projections on either side of attention ("DeepSeek V4.1-Flash. Every layer, connected",
 * "The query and output paths": low-rank query projection, grouped output projection;
 * "DeepSeek V4 Inside": query rank 1024, RMSNorm on the query head, 64 heads in 8 output
 * groups).  RMSNorm(v) = v / sqrt(mean(v^2) + eps) over the last axis.
 *
 * csa2_query_proj - the attention query of hidden states x:
 *   c   = W_DQ x                          (hidden -> q_rank)
 *   c   = RMSNorm(c) * g_q
 *   q   = W_UQ c                          (q_rank -> n_heads x 512)
 *   q_h = RMSNorm(q_h) * g_head           per head, one gain vector shared by the heads
 * The rotation of the head's last 64 coordinates is attention's (csa2_sparse_attn).
 * Tensor cores, bf16 inputs, fp32 accumulation; c is held in bf16 as c * g_q with its
 * RMSNorm factor applied to the up-projection's fp32 result.  Two kernel launches.
 * ------------------------------------------------------------------------------------ */
typedef struct {
  int32_t n_tokens;           /* T >= 0 */
  int32_t hidden;             /* multiple of 64 */
  int32_t q_rank;             /* multiple of 128 */
  int32_t n_heads;            /* >= 1 (heads of 512) */
  const void* x;              /* [T, hidden] bf16 */
  const void* w_dq;           /* [q_rank, hidden] bf16 (row f = the weights of feature f) */
  const float* g_q;           /* [q_rank] or NULL (gain 1) */
  const void* w_uq;           /* [n_heads * 512, q_rank] bf16 */
  const float* g_head;        /* [512] or NULL (gain 1) */
  float eps;                  /* >= 0 */
  void* q;                    /* out [T, n_heads, 512] bf16 */
  void* workspace;            /* csa2_query_proj_workspace_size bytes, any contents */
  size_t workspace_bytes;
  int32_t* dev_status;        /* optional device int32: CSA2_ETIMEOUT when a bounded wait on the
                                 tensor cores gave up (outputs then undefined); or NULL */
} csa2_query_proj_args;

/* Pointers device; x, the weights, q and workspace 16-byte aligned. */
size_t csa2_query_proj_workspace_size(const csa2_query_proj_args* a);
csa2_status csa2_query_proj(const csa2_query_proj_args* a, void* stream);

/* ------------------------------------------------------------------------------------
 * csa2_out_proj - grouped low-rank output projection of attention's output o (taken after
 * attention's inverse rotation): the heads split into n_groups groups of consecutive heads;
 *   y_g = W_OA[g] concat(o_h, h in group g)    (n_heads / n_groups * 512 -> o_rank)
 *   out = W_OB concat(y_0, .., y_{G-1})        (n_groups * o_rank -> hidden)
 * Tensor cores, bf16 inputs, fp32 accumulation, y held in bf16.  Two kernel launches.
 * ------------------------------------------------------------------------------------ */
typedef struct {
  int32_t n_tokens;           /* T >= 0 */
  int32_t n_heads;            /* multiple of n_groups */
  int32_t n_groups;           /* >= 1 */
  int32_t o_rank;             /* multiple of 128 */
  int32_t hidden;             /* multiple of 128 */
  const void* o;              /* [T, n_heads, 512] bf16 */
  const void* w_oa;           /* [n_groups, o_rank, n_heads / n_groups * 512] bf16 */
  const void* w_ob;           /* [hidden, n_groups * o_rank] bf16 */
  void* out;                  /* out [T, hidden] bf16 */
  void* workspace;            /* csa2_out_proj_workspace_size bytes, any contents */
  size_t workspace_bytes;
  int32_t* dev_status;        /* as in csa2_query_proj_args */
} csa2_out_proj_args;

/* Pointers device, 16-byte aligned. */
size_t csa2_out_proj_workspace_size(const csa2_out_proj_args* a);
csa2_status csa2_out_proj(const csa2_out_proj_args* a, void* stream);

/* ------------------------------------------------------------------------------------
 * csa2_expand_mxfp4 - MXFP4 indexer keys (OCP Microscaling: blocks of 32 E2M1 elements with
 * one UE8M0 exponent; "DeepSeek-V4.1-Flash explained", section 7 table) to their bf16 values,
 * out[j, d] = level(j, d) * 2^(e(j, d / 32) - 127): exact (every such value is a bf16 value;
 * e = 255 gives NaN).  A prefill chunk reuses its keys for every query, so it expands them
 * once and runs csa2_index_scores on the bf16 copy (the tensor-core prefill GEMM).
 * ------------------------------------------------------------------------------------ */
typedef struct {
  int64_t n_records;          /* records (all sequences) */
  const void* codes;          /* [n_records, 64] uint8, two E2M1 codes per byte, low nibble first */
  const void* exps;           /* [n_records, 4] uint8 */
  void* out;                  /* out [n_records, 128] bf16 */
} csa2_expand_args;

/* Pointers device; codes and out 16-byte aligned. */
csa2_status csa2_expand_mxfp4(const csa2_expand_args* a, void* stream);

/* ------------------------------------------------------------------------------------
 * csa2_linear - one plain projection out = x W^T on the tensor cores (bf16 inputs, fp32
 * accumulation, bf16 output rounded to nearest even): the building block of the path's
 * other linear maps, e.g. the encoder's indexer keys derived from its compressed entries
 * ("DeepSeek V4.1-Flash. Every layer, connected", "The global and index paths": indexer
 * keys come from the main KV).  One kernel launch.
 * ------------------------------------------------------------------------------------ */
typedef struct {
  int32_t n_tokens;           /* T >= 0 */
  int32_t in_features;        /* multiple of 64 */
  int32_t out_features;       /* multiple of 128 */
  const void* x;              /* [T, in_features] bf16 */
  const void* w;              /* [out_features, in_features] bf16 */
  void* out;                  /* out [T, out_features] bf16 */
  int32_t* dev_status;        /* as in csa2_query_proj_args */
} csa2_linear_args;

/* Pointers device, 16-byte aligned. */
csa2_status csa2_linear(const csa2_linear_args* a, void* stream);

/* ------------------------------------------------------------------------------------
 * Utilities
 * ------------------------------------------------------------------------------------ */
const char* csa2_status_string(csa2_status s);
/* Copies the device status word written by kernels (device index checks) to the host.
 * Synchronizes `stream` first.  Returns CSA2_OK and stores the word in *host_out. */
csa2_status csa2_read_device_status(const int32_t* dev_status, int32_t* host_out, void* stream);
/* Library version, e.g. 0x000100 for 0.1.0. */
int32_t csa2_version(void);

/* Overrides of the launch heuristics, process-wide, for tests and tuning.  By default every
 * call chooses its launch shapes from the problem's shapes and the device; results do not
 * depend on these settings beyond the fp32 summation order of csa2_query_proj /
 * csa2_out_proj / csa2_linear.  Not thread-safe with respect to calls in flight on the host
 * (a call reads each setting once). */
typedef enum csa2_tuning {
  CSA2_TUNE_SCAN_SEGMENTS = 0,  /* segments per row of an indexer scan; 0 = automatic, 1..64 */
  CSA2_TUNE_SCAN_WARP_MMA = 1,  /* 1: every scan takes the warp-MMA kernel; 0 = automatic */
  CSA2_TUNE_SCAN_CLUSTER = 2,   /* 0: the tcgen05 decode scan's segments merge through lists
                                   instead of selecting as a cluster; 1 = automatic (default) */
  CSA2_TUNE_PROJ_KSPLIT = 3,    /* K split of the projection GEMMs, 1..8; 0 = automatic */
  CSA2_TUNE_ATTN_ROWS = 4,      /* attention kernel: 1 = a block per (row, 128-entry tile) and a
                                   merge kernel; 2 / 3 = a block per (row, 32 / 16 heads) over all
                                   of the row's tiles; 4 = a block per (row, 32 heads) with the
                                   tiles' copies and arithmetic pipelined (bf16 latents and window
                                   only, otherwise 1); 0 = automatic (4 for at least two rows per
                                   SM with bf16 latents and window, else 1) */
  CSA2_TUNE_COUNT = 5
} csa2_tuning;
/* Returns CSA2_EINVAL for an unknown knob or a value outside its range. */
csa2_status csa2_set_tuning(int32_t knob, int32_t value);

/* Self-test of the bounded device wait the tensor-core kernels use (no counterpart in the
 * pages: failure handling of this library).  Launches one block that waits, `tries` times
 * (1 .. 2^20), on an mbarrier nothing signals; the wait gives up and stores CSA2_ETIMEOUT in
 * the device int32 *dev_status, as the kernels do, and the block returns normally.  Returns
 * CSA2_EINVAL for a NULL dev_status or tries out of range, CSA2_ECUDA for a failed launch. */
csa2_status csa2_selftest_wait_timeout(int32_t* dev_status, int32_t tries, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H */
