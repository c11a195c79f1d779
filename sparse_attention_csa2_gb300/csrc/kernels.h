// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace csa2 {

// Multiprocessors of the current device (queried once per device).
int device_sm_count();
// Current value of a launch-heuristic override (csa2_tuning in csa2.h).
int tuning(int knob);

// Indexer scan over one query row per grid row, n_seg segments per row.
struct ScanParams {
  const void* q_idx;          // [n_rows, 32, 128] bf16
  const float* w;             // [n_rows, 32]
  const void* k_idx;          // [n_seq, N, 128] bf16 | E4M3
  const float* k_scale;       // [n_seq, N] (FP8)
  long long N;
  const int32_t* seq_of_row;
  const int32_t* n_visible;
  const int32_t* cand;        // gather mode: [n_rows, cand_stride]
  const int32_t* n_cand;
  long long cand_stride;
  int cand_run;               // tcgen05 decode over candidates: they come in runs of cand_run
                              // consecutive positions (a multiple of 64) from the pool's blocks
  int n_rows;
  int unit;                   // entries per scheduling unit (16, or block_size with block_max)
  float* scores;              // optional [n_rows, scores_stride]
  long long scores_stride;
  long long scores_len;       // columns to fill (-inf past the candidates)
  float* block_max;           // optional [n_rows, bmax_stride]
  long long bmax_stride;
  long long n_blocks;
  int K;                      // 0 = no top-K
  int32_t* idx;               // final [n_rows, K] when n_seg == 1
  uint32_t* seg_keys;         // [n_rows, n_seg, K] when n_seg > 1
  int32_t* seg_pos;
  int32_t* seg_cnt;           // [n_rows, n_seg]
  uint32_t* seg_thr;          // [n_rows, n_seg] K-th key of each full segment list, else 0
  unsigned long long* row_done;  // tcgen05 decode: [n_rows] (call tag << 32 | finished segments);
                                 // the last segment of a row to finish merges the row's lists
  uint32_t call_tag;             // differs between consecutive calls (no clearing of row_done)
  int cluster_merge;             // tcgen05 decode: the segments of a row form a cluster and
                                 // select the row's top-K together (no lists, no merge)
  int32_t* dev_status;        // optional: CSA2_ETIMEOUT when a bounded wait gives up
  int pdl_trigger;            // set by the launcher: the grid is one wave, so a kernel launched
                              // after it with programmatic dependent launch may start early
  int seg_table;              // set by the launcher: entries of the per-segment block table
  int fast_select;            // set by the launcher (cluster selection): candidates are marked
                              // during the stream against a running bound, and one block of the
                              // cluster selects among them after it
};

// key format of the warp-MMA scan: 0 bf16, 1 FP8 rows, 2 MXFP4
size_t scan_smem_bytes(int fmt, int K);

// tcgen05 indexer: decode rows (bf16 or FP8 keys, records in place) and prefill tiles (bf16).
bool mma_indexer_available();
// Tensor map of a row-major bf16 matrix [rows x cols] (rows row_bytes apart): boxes of 64
// columns x box_rows rows in the 128-byte swizzle, zeros outside the matrix.
bool make_tmap_bf16(CUtensorMap* tm, const void* base, unsigned long long cols, unsigned long long rows,
                    unsigned long long row_bytes, unsigned box_rows);
int mma_decode_max_seg_blocks();
int mma_decode_max_segment();  // most records one decode segment may hold
bool mma_decode_can_merge(int n_seg, int K);  // the decode scan can merge its segments' lists itself
bool mma_decode_cluster_ok(int n_seg, int n_rows, int K, int max_seg_blocks, bool fp8);  // segments of a row as a cluster
cudaError_t launch_mma_decode(const ScanParams& p, long long n_seq_rows, int n_seg, int max_seg_blocks, bool fp8,
                              cudaStream_t stream);
cudaError_t launch_mma_prefill(const ScanParams& p, int n_ctas, int n_parts, cudaStream_t stream);
cudaError_t launch_index_scan(const ScanParams& p, int fmt, bool gather, int n_seg, cudaStream_t stream);
// tcgen05 FP8 decode scan with the streaming top-K engine (two blocks per SM): FULL rows of
// any length, top-K of at most kEngMaxK, no block maxima, candidates or scores.
bool fp8_stream_ok(int K);
cudaError_t launch_fp8_stream(const ScanParams& p, long long n_seq_rows, int n_seg, cudaStream_t stream);

// Streaming top-K over per-row entry streams (scores, or the lists of earlier segments).
struct FeedParams {
  int n_rows;
  int K;
  // source A: scores[row, j], j < n_valid[row]; position cand[row, j] or j
  const float* scores;
  long long scores_stride;
  const int32_t* n_valid;
  int valid_div;              // entries of row r: ceil(n_valid[r] / valid_div)
  const int32_t* cand;
  long long cand_stride;
  // source B: segment lists (key, pos) [n_rows, in_seg, in_K] with counts [n_rows, in_seg]
  const uint32_t* in_keys;
  const int32_t* in_pos;
  const int32_t* in_cnt;
  const uint32_t* in_thr;     // optional [n_rows, in_seg]: K-th key of each full list
  int in_seg;
  int in_K;
  // output: final idx [n_rows, K] (out_seg == 1) or lists [n_rows, out_seg, K]
  int32_t* idx;
  // optional, source A with out_seg == 1: the kept entries are blocks of pool_bs positions
  // (n_valid counts positions) and expand to pool [n_rows, K * pool_bs] (-1 past the visible
  // positions and for missing blocks) with n_pool [n_rows] valid positions
  int32_t* pool;
  int32_t* n_pool;
  int pool_bs;
  uint32_t* out_keys;
  int32_t* out_pos;
  int32_t* out_cnt;
  uint32_t* out_thr;
};

size_t feed_smem_bytes(int K);
int topk_segments(int n_rows, long long L);  // segments csa2_topk splits each row into
cudaError_t launch_topk_feed(const FeedParams& p, bool from_lists, int out_seg, cudaStream_t stream);
cudaError_t launch_lists_merge(const FeedParams& p, cudaStream_t stream);  // segment lists -> final idx
// Exact top-K of every row by multi-pass radix selection over the row in memory (source A
// with n_valid, optional cand; rows far longer than K), one block per row.
cudaError_t launch_row_topk(const FeedParams& p, cudaStream_t stream);
struct AttnParams {
  const void* q;
  const int64_t* q_pos;
  const int32_t* seq_of_row;
  int n_rows;
  long long N;
  const void* lat;
  const uint8_t* lat_scale;
  int lat_fmt;
  const int32_t* idx;
  int K;
  const void* swa;
  const float* swa_scale;
  int swa_fmt;
  long long swa_rows;
  const int64_t* swa_pos0;
  int window;
  const float* sink;
  float theta;
  float scale;
  double inv_freq[32];        // theta^(-2i/64), i = 0..31 (computed on the host in double)
  float* part_o;              // [n_rows, n_split, 64, 512]
  float* part_ml;             // [n_rows, n_split, 64, 2]
  // optional [n_rows, 64]: the row's rotary cos (0..31) and sin (32..63) at +q_pos, written by
  // one tile block per row for the merge (null: the merge computes them)
  float* rope_cs;
  // a device's share of a record-range split: idx holds global positions; those outside
  // [range_first, range_first + range_count) are skipped, the others index the latents at
  // position - range_first (range_count == 0: no range); skip_window masks the window entries
  long long range_first;
  long long range_count;
  int skip_window;
  // merge of partials from several parts (record ranges): part k's tiles of row r sit at
  // part_o + k * part_stride_o + (r * part_tiles + t) * 64 * 512 (part_ml likewise, 64 * 2
  // per tile); part_tiles == 0: one part of n_split tiles (the layout above)
  int part_tiles;
  long long part_stride_o;
  long long part_stride_ml;
  void* out;                  // fp32, or bf16 when out_bf16
  int out_bf16;
  float* sink_mass;
  int32_t* dev_status;        // optional: CSA2_EDEVICE_INDEX on an out-of-range record index
};

// Cache writer (csa2_write_records).
struct WriteParams {
  long long n_rows;
  const void* x;          // [n_rows, 512] float32 (x_f32) or bf16
  int x_f32;
  const int64_t* pos;     // [n_rows] or null (no rotation)
  double inv_freq[32];    // theta^(-2i/64), computed on the host in double
  const int64_t* dst_row; // [n_rows]
  long long cache_rows;
  int out_dtype;          // CSA2_FP4_E2M1_G16 / _G32 or CSA2_FP8_E4M3_ROWSCALE
  void* codes;
  void* scales;
  int32_t* dev_status;
};
cudaError_t launch_write_records(const WriteParams& p, cudaStream_t stream);
// MXFP4 records -> bf16 records (csa2_expand_mxfp4).
cudaError_t launch_expand_mxfp4(long long n_records, const void* codes, const void* exps, void* out,
                                cudaStream_t stream);
// Sequence compressor (csa2_compress).
cudaError_t launch_compress(long long n_entries, int ratio, const void* kv, const void* gate, bool x_f32, float* out,
                            cudaStream_t stream);

// Projections around attention (csa2_query_proj, csa2_out_proj): one tcgen05 GEMM
// out[t, f] = sum_k A[f, k] B[t, k] per launch, A = weights (features x K), B = activations
// (tokens x K), with the epilogue of `mode`.
enum ProjMode { kProjPlain = 0, kProjDown = 1, kProjUp = 2 };
constexpr int kProjMaxStages = 12;
struct ProjParams {
  int mode;
  int n_tok;
  int k_steps;                // K / 64 of one group
  int m_tiles;                // features of one group / 128
  int ks;                     // K splits, reduced across a cluster of ks blocks (1 for kProjUp)
  int bn;                     // token tile: 32, 64, 128 or 256
  int stages;
  int a_rows_per_group;       // A row offset of group g: g * a_rows_per_group
  int b_cols_per_group;       // B column offset of group g
  void* out;                  // bf16 [n_tok, out_ld]; group g's features start at column g * out_cols_per_group
  long long out_ld;
  int out_cols_per_group;
  const float* gain;          // kProjDown: [features]; kProjUp: [512], by feature % 512; null: 1
  float* ss;                  // kProjDown: out [m_tiles * ks, n_tok] sums of squares; kProjUp: in [ss_tiles, n_tok]
  int ss_tiles;
  float inv_rank;             // kProjUp: 1 / (rank of the low-rank vector)
  float eps;
  int32_t* dev_status;
};
size_t proj_smem_bytes(int bn, int stages);
// Bytes of the pipeline buffers the epilogue reuses (the staged output tile; with ks > 1 the
// rows received from the cluster's blocks).
size_t proj_epilogue_bytes(int bn, int ks);
cudaError_t launch_proj(const CUtensorMap& tmA, const CUtensorMap& tmB, const ProjParams& p, int groups,
                        cudaStream_t stream);

int attn_smem_bytes();
cudaError_t launch_sparse_attn(const AttnParams& p, int n_split, cudaStream_t stream);
// The tile kernel alone (partials of n_split tiles per row) and the merge alone (n_tiles
// partials per row in the layout p describes, sink, normalisation, inverse RoPE).
cudaError_t launch_attn_tiles(const AttnParams& p, int n_split, cudaStream_t stream);
cudaError_t launch_attn_merge(const AttnParams& p, int n_tiles, cudaStream_t stream);
// Candidate lists of a record range: from the selected columns idx [n_rows, K] (-1 padded) of
// scores [n_rows, stride], writes scores and positions (offset + column) of the selected
// entries, -inf / -1 padded, and their count per row.
cudaError_t launch_shard_list(int n_rows, int K, const int32_t* idx, const float* scores, long long stride,
                              long long offset, float* out_scores, int32_t* out_pos, int32_t* out_cnt,
                              cudaStream_t stream);
// Gathered candidate lists (list-major scores / positions [n_lists, n_rows, k_in], counts
// [n_lists, n_rows]) to the list merge's row-major keys, positions and counts.
cudaError_t launch_lists_to_rows(int n_rows, int n_lists, int k_in, const float* scores, const int32_t* pos,
                                 const int32_t* cnt, uint32_t* keys, int32_t* pos_out, int32_t* cnt_out,
                                 cudaStream_t stream);

}  // namespace csa2
