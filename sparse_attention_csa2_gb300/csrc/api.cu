// The C ABI of the CSA2 attention step (include/csa2.h): host-side validation, workspace
// layout, work decomposition and launch sequencing.  Nothing here synchronizes or allocates.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstring>

#include "../../include/csa2.h"
#include "kernels.h"

namespace csa2 {

// Multiprocessor count per device, queried once per device (launch plans are sized by it on
// every call).
int device_sm_count() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cached[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 0 && dev < kMaxDev) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  if (dev >= 0 && dev < kMaxDev) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Process-wide overrides of the launch heuristics (csa2_set_tuning); the defaults mean
// "chosen per call from the shapes and the device".
namespace {
std::atomic<int> g_tuning[CSA2_TUNE_COUNT] = {{0}, {0}, {1}, {0}, {0}};
}  // namespace

int tuning(int knob) { return g_tuning[knob].load(std::memory_order_relaxed); }

namespace {

// Tag of one fused decode call for the scan's per-row completion counters: consecutive calls
// get different tags, so a counter left by an earlier call (or never written) is recognised
// and restarted instead of being cleared before every call.  Starts from a clock reading so
// that a workspace shared across processes is unlikely to hold a matching stale tag.
uint32_t next_call_tag() {
  static std::atomic<uint32_t> tag{static_cast<uint32_t>(
      std::chrono::steady_clock::now().time_since_epoch().count() * 2654435761ull)};
  return tag.fetch_add(1, std::memory_order_relaxed) + 1;
}

constexpr int kScanMaxK = 512;  // per-warp survivor buffers of the fused scan fit K <= 512

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool pow2(long long v) { return v > 0 && (v & (v - 1)) == 0; }
size_t align_up(size_t v, size_t a = 256) { return (v + a - 1) / a * a; }

int sm_count() { return device_sm_count(); }

// Segments per row of the indexer scan: one resident block per SM, one wave; every segment
// keeps at least min_seg records (4096 for full scans) so the per-segment top-K and pipeline
// start-up stay small.
int scan_segments(int n_rows, long long L, long long min_seg = 4096) {
  const int forced = tuning(CSA2_TUNE_SCAN_SEGMENTS);
  if (forced > 0) return forced;
  const int slots = sm_count();
  if (n_rows >= slots) return 1;
  long long s = slots / (n_rows > 0 ? n_rows : 1);
  const long long cap = L / min_seg;
  if (s > cap) s = cap;
  if (s > 64) s = 64;
  return s < 1 ? 1 : (int)s;
}

// Tiles of 128 attended entries per row: one attention block each (K + window <= 2048, so
// at most 16).
int attn_splits(int n_rows, int K, int window) {
  (void)n_rows;
  const int n_tiles = (K + window + 127) / 128;
  return n_tiles < 1 ? 1 : n_tiles;
}

csa2_status cuda_status(cudaError_t e) { return e == cudaSuccess ? CSA2_OK : CSA2_ECUDA; }

// Which indexer kernel runs a scan: the tcgen05 decode kernel takes bf16 or FP8 keys read in
// place, the tcgen05 prefill kernel bf16 keys; other FP8 scans and candidate lists not in runs
// of 64 records take the warp-MMA scan.
enum class ScanPath { kWarpMma, kTc05Decode, kTc05Prefill, kTc05Stream };

// cand_run: the candidates come in runs of that many consecutive records (a Reindex pool of
// whole blocks); runs of a multiple of 64 let the tcgen05 scan load them with TMA.
// stream_k: the top-K of a FULL decode layer (no block maxima), which the streaming FP8 scan
// can take; 0 otherwise.
int tc05_segments(int n_rows, long long L, int unit, long long min_seg = 4096);

ScanPath scan_path(const csa2_index_args* a, bool want_topk, int cand_run = 0, int stream_k = 0) {
  if (!mma_indexer_available() || tuning(CSA2_TUNE_SCAN_WARP_MMA) != 0 || a->k_dtype == CSA2_MXFP4)
    return ScanPath::kWarpMma;
  if (a->cand != nullptr && !(want_topk && cand_run > 0 && cand_run % 64 == 0)) return ScanPath::kWarpMma;
  const bool fp8 = a->k_dtype == CSA2_FP8_E4M3_ROWSCALE;
  if (!want_topk && a->block_max == nullptr && a->n_seq == 1 && a->n_rows >= 64)
    return fp8 ? ScanPath::kWarpMma : ScanPath::kTc05Prefill;
  if (fp8) {
    // The decode kernel keeps every key of a segment in shared memory, one block per SM, so
    // it takes FP8 rows only where its grid is one wave (a second, partial wave of 16K-record
    // segments costs more than one wave of longer segments elsewhere).  Longer FULL rows take
    // the streaming FP8 scan (bounded top-K buffers, two blocks per SM), else the warp-MMA scan.
    const long long L = a->cand != nullptr ? a->L : a->n_records;
    if ((long long)a->n_rows * tc05_segments(a->n_rows, L, 128) > sm_count())
      return want_topk && stream_k > 0 && a->cand == nullptr && fp8_stream_ok(stream_k) ? ScanPath::kTc05Stream
                                                                                       : ScanPath::kWarpMma;
  }
  return ScanPath::kTc05Decode;
}

// Segments per row for the tcgen05 decode scan: whole waves of resident blocks, each
// segment's blocks (for the block maxima) within the kernel's shared-memory table.
int tc05_segments(int n_rows, long long L, int unit, long long min_seg) {
  int n = scan_segments(n_rows, L, min_seg);
  const long long units = (L + unit - 1) / unit;
  const int max_blocks = mma_decode_max_seg_blocks();
  const long long max_units = mma_decode_max_segment() / unit;  // a segment's keys fit in shared memory
  while ((units + n - 1) / n > max_blocks || (units + n - 1) / n > max_units) ++n;
  return n;
}

// Segments per row for the streaming FP8 scan: two resident blocks per SM, at most 128 lists
// per row (the lists merge's table), none shorter than 2,048 records.
int stream_segments(int n_rows, long long L) {
  const int forced = tuning(CSA2_TUNE_SCAN_SEGMENTS);
  if (forced > 0) return forced;
  long long s = 2LL * sm_count() / (n_rows > 0 ? n_rows : 1);
  s = std::min(s, std::max(1LL, L / 2048));
  s = std::min(s, 128LL);
  return s < 1 ? 1 : (int)s;
}

cudaError_t launch_scan(ScanParams& p, const csa2_index_args* a, bool want_topk, int n_seg, cudaStream_t s,
                        int stream_k = 0) {
  switch (scan_path(a, want_topk, p.cand_run, stream_k)) {
    case ScanPath::kTc05Stream:
      return launch_fp8_stream(p, (long long)a->n_seq * a->n_records, n_seg, s);
    case ScanPath::kTc05Prefill: {
      // work items: (8-query tile, share of its key tiles); enough items to balance the
      // persistent grid, none shorter than ~16 key tiles
      const int n_qt = (p.n_rows + 7) / 8;
      const int ctas = sm_count();
      const long long tiles = (a->n_records + 127) / 128;
      int parts = 1;
      while (n_qt * parts < 6 * ctas && tiles / (2 * parts) >= 16 && parts < 64) parts *= 2;
      return launch_mma_prefill(p, ctas, parts, s);
    }
    case ScanPath::kTc05Decode: {
      // shared-memory table per segment: block maxima, or the candidates' 64-slot run starts
      const int seg_blocks =
          p.block_max ? (int)(((a->n_records + p.unit - 1) / p.unit + n_seg - 1) / n_seg)
          : p.cand   ? (int)(2 * (((a->L + p.unit - 1) / p.unit + n_seg - 1) / n_seg))
                     : 0;
      return launch_mma_decode(p, (long long)a->n_seq * a->n_records, n_seg, seg_blocks,
                               a->k_dtype == CSA2_FP8_E4M3_ROWSCALE, s);
    }
    default:
      return launch_index_scan(p, a->k_dtype == CSA2_FP8_E4M3_ROWSCALE ? 1 : a->k_dtype == CSA2_MXFP4 ? 2 : 0,
                               a->cand != nullptr, n_seg, s);
  }
}

// ---- workspace carving
struct Carve {
  uint8_t* base;
  size_t off = 0;
  template <class T>
  T* take(size_t count) {
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off = align_up(off + count * sizeof(T));
    return p;
  }
};

// ------------------------------------------------------------------ index validation
csa2_status check_index(const csa2_index_args* a, bool need_outputs) {
  if (!a) return CSA2_EINVAL;
  if (a->n_rows < 0 || a->n_seq < 1 || a->n_records < 1 || a->n_records > (1LL << 31) - 1) return CSA2_EINVAL;
  if (a->n_rows == 0) return CSA2_OK;
  if (!a->q_idx || !a->w || !a->k_idx || !a->seq_of_row || !a->n_visible) return CSA2_EINVAL;
  if (!aligned(a->q_idx, 16) || !aligned(a->k_idx, 16) || !aligned(a->w, 4)) return CSA2_EINVAL;
  if (a->k_dtype != CSA2_BF16 && a->k_dtype != CSA2_FP8_E4M3_ROWSCALE && a->k_dtype != CSA2_MXFP4)
    return CSA2_EINVAL;
  if (a->k_dtype != CSA2_BF16 && (!a->k_scale || !aligned(a->k_scale, 4))) return CSA2_EINVAL;
  if (a->cand) {
    if (!a->n_cand || a->L < 1 || a->L > (1LL << 31) - 1) return CSA2_EINVAL;
  }
  if (need_outputs && !a->scores && !a->block_max) return CSA2_EINVAL;
  if (a->block_max) {
    if (a->cand) return CSA2_EINVAL;
    if (!pow2(a->block_size) || a->block_size < 16 || a->block_size > 4096) return CSA2_EUNSUPPORTED;
  }
  return CSA2_OK;
}

ScanParams scan_params(const csa2_index_args* a) {
  ScanParams p{};
  p.q_idx = a->q_idx;
  p.w = a->w;
  p.k_idx = a->k_idx;
  p.k_scale = a->k_scale;
  p.N = a->n_records;
  p.seq_of_row = a->seq_of_row;
  p.n_visible = a->n_visible;
  p.cand = a->cand;
  p.n_cand = a->n_cand;
  p.cand_stride = a->cand ? a->L : 0;
  p.n_rows = a->n_rows;
  p.unit = 16;
  return p;
}

// ------------------------------------------------------------------ attention validation
csa2_status check_attn(const csa2_attn_args* a, bool need_idx, bool need_out = true) {
  if (!a) return CSA2_EINVAL;
  if (a->n_rows < 0 || a->n_seq < 1 || a->n_records < 1 || a->n_records > (1LL << 31) - 1) return CSA2_EINVAL;
  if (a->n_rows == 0) return CSA2_OK;
  if (!a->q || !a->q_pos || !a->seq_of_row || !a->swa_pos0) return CSA2_EINVAL;
  if (need_out && (!a->sink || !a->out)) return CSA2_EINVAL;
  if (a->K < 0 || a->K > CSA2_MAX_TOPK || a->window < 0 || a->window > 1024) return CSA2_EUNSUPPORTED;
  if (a->K + a->window < 1) return CSA2_EINVAL;
  if (a->K > 0 && (!a->latents || (need_idx && !a->idx))) return CSA2_EINVAL;
  if (!aligned(a->q, 16) || (need_out && !aligned(a->out, 16)) || (a->latents && !aligned(a->latents, 16)))
    return CSA2_EINVAL;
  if (a->lat_dtype == CSA2_FP4_E2M1_G32 || a->lat_dtype == CSA2_FP4_E2M1_G16) {
    if (a->K > 0 && !a->lat_scale) return CSA2_EINVAL;
  } else if (a->lat_dtype != CSA2_BF16) {
    return CSA2_EINVAL;
  }
  if (a->window > 0) {
    if (!a->swa || !aligned(a->swa, 16) || a->swa_rows < 1) return CSA2_EINVAL;
    if (a->swa_dtype == CSA2_FP8_E4M3_ROWSCALE) {
      if (!a->swa_scale) return CSA2_EINVAL;
    } else if (a->swa_dtype != CSA2_BF16) {
      return CSA2_EINVAL;
    }
  }
  if (!(a->rope_theta > 0.f)) return CSA2_EINVAL;
  return CSA2_OK;
}

AttnParams attn_params(const csa2_attn_args* a, const int32_t* idx) {
  AttnParams p{};
  p.q = a->q;
  p.q_pos = a->q_pos;
  p.seq_of_row = a->seq_of_row;
  p.n_rows = a->n_rows;
  p.N = a->n_records;
  p.lat = a->latents;
  p.lat_scale = a->lat_scale;
  p.lat_fmt = a->lat_dtype;
  p.idx = idx;
  p.K = a->K;
  p.swa = a->swa;
  p.swa_scale = a->swa_scale;
  p.swa_fmt = a->swa_dtype;
  p.swa_rows = a->swa_rows;
  p.swa_pos0 = a->swa_pos0;
  p.window = a->window;
  p.sink = a->sink;
  p.theta = a->rope_theta;
  p.scale = a->softmax_scale;
  for (int i = 0; i < CSA2_ROPE_DIM / 2; ++i)
    p.inv_freq[i] = std::pow((double)a->rope_theta, -2.0 * i / (double)CSA2_ROPE_DIM);
  p.out = a->out;
  p.out_bf16 = a->out_bf16 != 0;
  p.sink_mass = a->sink_mass;
  p.dev_status = a->dev_status;
  return p;
}

// attention partials (O, then m and l per tile and head) and each row's rotary cos / sin
size_t attn_workspace(const csa2_attn_args* a, int n_split) {
  return align_up((size_t)a->n_rows * n_split * CSA2_HEADS * CSA2_HEAD_DIM * 4) +
         align_up((size_t)a->n_rows * n_split * CSA2_HEADS * 2 * 4) + align_up((size_t)a->n_rows * CSA2_ROPE_DIM * 4);
}

csa2_status run_attn(const csa2_attn_args* a, const int32_t* idx, uint8_t* ws, cudaStream_t s) {
  const int n_split = attn_splits(a->n_rows, a->K, a->window);
  AttnParams p = attn_params(a, idx);
  Carve c{ws};
  p.part_o = c.take<float>((size_t)a->n_rows * n_split * CSA2_HEADS * CSA2_HEAD_DIM);
  p.part_ml = c.take<float>((size_t)a->n_rows * n_split * CSA2_HEADS * 2);
  p.rope_cs = c.take<float>((size_t)a->n_rows * CSA2_ROPE_DIM);
  return cuda_status(launch_sparse_attn(p, n_split, s));
}

// ------------------------------------------------------------------ projections
// Launch shape of one projection GEMM: token tile bn (the MMA's N), pipeline stages and the
// K split ks (a cluster of ks blocks per tile).  The split is the smallest that gives 1.5
// blocks per SM for narrow token tiles (two fit on an SM) and 3/4 for wide ones, capped at 8:
// HBM streaming wants every SM busy, and two blocks per SM, each with its own pipeline, hid the
// load latency better than one with twice the stages (decode output projection: 45.6 against
// 47.6 us); every split adds a distributed-shared-memory exchange.  A grid that fits on the
// SMs runs one block per SM with a deep pipeline (~200 KB of loads in flight per SM); a larger
// one two blocks per SM with half the stages each, so that one block's epilogue overlaps the
// other's main loop (prefill, 256-token tiles: 0.92 -> 0.73 ms for the four GEMMs).
struct ProjPlan {
  int bn, stages, ks;
};

int proj_bn(int n_tok) { return n_tok <= 32 ? 32 : n_tok <= 64 ? 64 : n_tok <= 128 ? 128 : 256; }

// tiles: blocks of one K split (feature tiles x token tiles x groups)
ProjPlan proj_plan(int n_tok, int k_steps, int tiles, bool allow_split) {
  const int bn = proj_bn(n_tok);
  const size_t stage = 128 * 128 + (size_t)bn * 128;
  const int sms = sm_count();
  int ks = 1;
  const int forced = tuning(CSA2_TUNE_PROJ_KSPLIT);
  if (forced > 0) {
    while (ks * 2 <= forced && ks < 8) ks *= 2;
  } else {
    // narrow token tiles (two blocks fit on an SM) aim for 1.5 blocks per SM, wide ones for 3/4
    const long long target4 = bn <= 64 ? 6LL * sms : 3LL * sms;  // 4 x the block target
    while (allow_split && ks < 8 && (long long)tiles * ks * 4 < target4) ks *= 2;
    // an 8-block cluster's exchange costs more than it gains unless a split of 4 leaves more
    // than half the SMs idle (decode: the final output stage 47.4 us at 8 against 45.6 at 4;
    // the 8 tiles of the down-projection 31.3 at 8 against 33.3 at 4)
    if (ks == 8 && (long long)tiles * 4 * 2 >= sms) ks = 4;
  }
  if (!allow_split) ks = 1;
  while (ks > 1 && ks > k_steps) ks /= 2;
  const bool two_per_sm = (long long)tiles * ks > sms;
  const size_t budget = two_per_sm ? 100 * 1024 : 200 * 1024;
  int stages = (int)std::min<size_t>(kProjMaxStages, budget / stage);
  while ((size_t)stages * stage < proj_epilogue_bytes(bn, ks) && stages < kProjMaxStages) ++stages;
  return ProjPlan{bn, stages, ks};
}

// ------------------------------------------------------------------ top-K plumbing
struct TopkPlan {
  int n_seg;
};

TopkPlan topk_plan(int n_rows, long long L) {
  TopkPlan t{1};
  const int slots = sm_count();
  if (n_rows < slots) {
    long long s = slots / (n_rows > 0 ? n_rows : 1);
    const long long by_len = (L + 8191) / 8192;
    if (s > by_len) s = by_len;
    if (s > 64) s = 64;
    t.n_seg = s < 1 ? 1 : (int)s;
  }
  return t;
}

size_t lists_bytes(int n_rows, int n_seg, int K) {
  if (n_seg <= 1) return 0;
  return 2 * align_up((size_t)n_rows * n_seg * K * 4) + 2 * align_up((size_t)n_rows * n_seg * 4);
}

}  // namespace

int topk_segments(int n_rows, long long L) { return topk_plan(n_rows, L).n_seg; }

}  // namespace csa2

using namespace csa2;

extern "C" {

const char* csa2_status_string(csa2_status s) {
  switch (s) {
    case CSA2_OK: return "ok";
    case CSA2_EINVAL: return "invalid argument";
    case CSA2_EUNSUPPORTED: return "unsupported size or format";
    case CSA2_ECUDA: return "CUDA launch or runtime error";
    case CSA2_ETIMEOUT: return "device-side wait timed out";
    case CSA2_EWORKSPACE: return "workspace missing or too small";
    case CSA2_EDEVICE_INDEX: return "device index out of range";
  }
  return "unknown status";
}

int32_t csa2_version(void) { return 0x000100; }

csa2_status csa2_set_tuning(int32_t knob, int32_t value) {
  if (knob < 0 || knob >= CSA2_TUNE_COUNT || value < 0) return CSA2_EINVAL;
  if (knob == CSA2_TUNE_SCAN_SEGMENTS && value > 64) return CSA2_EINVAL;
  if (knob == CSA2_TUNE_PROJ_KSPLIT && value > 8) return CSA2_EINVAL;
  if (knob == CSA2_TUNE_ATTN_ROWS && value > 4) return CSA2_EINVAL;
  g_tuning[knob].store(value, std::memory_order_relaxed);
  return CSA2_OK;
}

csa2_status csa2_read_device_status(const int32_t* dev_status, int32_t* host_out, void* stream) {
  if (!dev_status || !host_out) return CSA2_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_out, dev_status, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return CSA2_ECUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? CSA2_OK : CSA2_ECUDA;
}

// ---------------------------------------------------------------------- index scores
csa2_status csa2_index_scores(const csa2_index_args* a, void* stream) {
  csa2_status st = check_index(a, true);
  if (st != CSA2_OK || a->n_rows == 0) return st;
  ScanParams p = scan_params(a);
  const long long L = a->cand ? a->L : a->n_records;
  p.scores = a->scores;
  p.scores_stride = L;
  p.scores_len = L;
  if (a->block_max) {
    p.block_max = a->block_max;
    p.n_blocks = (a->n_records + a->block_size - 1) / a->block_size;
    p.bmax_stride = p.n_blocks;
    p.unit = a->block_size;
  }
  p.K = 0;
  const ScanPath path = scan_path(a, false);
  if (path == ScanPath::kTc05Decode && !a->block_max) p.unit = 128;
  const int n_seg = path == ScanPath::kTc05Decode ? tc05_segments(a->n_rows, L, p.unit) : scan_segments(a->n_rows, L);
  return cuda_status(launch_scan(p, a, false, n_seg, static_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------------- top-K
size_t csa2_topk_workspace_size(const csa2_topk_args* a) {
  if (!a || a->n_rows <= 0 || a->K < 1) return 0;
  const TopkPlan t = topk_plan(a->n_rows, a->L);
  return lists_bytes(a->n_rows, t.n_seg, a->K);
}

csa2_status csa2_topk(const csa2_topk_args* a, void* stream) {
  if (!a || a->n_rows < 0) return CSA2_EINVAL;
  if (a->n_rows == 0) return CSA2_OK;
  if (!a->scores || !a->n_valid || !a->idx || a->L < 1 || a->L > (1LL << 24)) return CSA2_EINVAL;
  if (a->K < 1 || a->K > CSA2_MAX_TOPK) return CSA2_EUNSUPPORTED;
  const size_t need = csa2_topk_workspace_size(a);
  if (need > 0 && (!a->workspace || a->workspace_bytes < need)) return CSA2_EWORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const TopkPlan t = topk_plan(a->n_rows, a->L);
  FeedParams f{};
  f.n_rows = a->n_rows;
  f.K = a->K;
  f.scores = a->scores;
  f.scores_stride = a->L;
  f.n_valid = a->n_valid;
  f.valid_div = 1;
  f.cand = a->cand;
  f.cand_stride = a->L;
  if (t.n_seg == 1) {
    f.idx = a->idx;
    // rows far longer than K (a prefill chunk's): radix selection over the row in memory;
    // otherwise the streaming engine
    if (a->L >= 8LL * a->K) return cuda_status(launch_row_topk(f, s));
    return cuda_status(launch_topk_feed(f, false, 1, s));
  }
  Carve c{static_cast<uint8_t*>(a->workspace)};
  f.out_keys = c.take<uint32_t>((size_t)a->n_rows * t.n_seg * a->K);
  f.out_pos = c.take<int32_t>((size_t)a->n_rows * t.n_seg * a->K);
  f.out_cnt = c.take<int32_t>((size_t)a->n_rows * t.n_seg);
  f.out_thr = c.take<uint32_t>((size_t)a->n_rows * t.n_seg);
  cudaError_t e = launch_topk_feed(f, false, t.n_seg, s);
  if (e != cudaSuccess) return CSA2_ECUDA;
  FeedParams m{};
  m.n_rows = a->n_rows;
  m.K = a->K;
  m.in_keys = f.out_keys;
  m.in_pos = f.out_pos;
  m.in_cnt = f.out_cnt;
  m.in_thr = f.out_thr;
  m.in_seg = t.n_seg;
  m.in_K = a->K;
  m.idx = a->idx;
  return cuda_status(launch_lists_merge(m, s));
}

// ---------------------------------------------------------------------- block pool
static size_t block_pool_ws(int n_rows, int n_keep) { return align_up((size_t)n_rows * n_keep * 4); }

size_t csa2_block_pool_workspace_size(const csa2_block_pool_args* a) {
  if (!a || a->n_rows <= 0 || a->n_keep < 1) return 0;
  return block_pool_ws(a->n_rows, a->n_keep);
}

csa2_status csa2_block_pool(const csa2_block_pool_args* a, void* stream) {
  if (!a || a->n_rows < 0) return CSA2_EINVAL;
  if (a->n_rows == 0) return CSA2_OK;
  if (!a->block_max || !a->n_visible || !a->pool || !a->n_pool || a->n_blocks < 1) return CSA2_EINVAL;
  if (a->block_size < 1 || a->block_size > 4096 || a->n_keep < 1) return CSA2_EINVAL;
  if (a->n_keep > CSA2_MAX_TOPK || (long long)a->n_keep * a->block_size > (1LL << 20)) return CSA2_EUNSUPPORTED;
  const size_t need = csa2_block_pool_workspace_size(a);
  if (!a->workspace || a->workspace_bytes < need) return CSA2_EWORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* kept = static_cast<int32_t*>(a->workspace);
  FeedParams f{};
  f.n_rows = a->n_rows;
  f.K = a->n_keep;
  f.scores = a->block_max;
  f.scores_stride = a->n_blocks;
  f.n_valid = a->n_visible;
  f.valid_div = a->block_size;
  f.idx = kept;
  f.pool = a->pool;
  f.n_pool = a->n_pool;
  f.pool_bs = a->block_size;
  return cuda_status(launch_topk_feed(f, false, 1, s));
}

// ---------------------------------------------------------------------- sparse attention
size_t csa2_sparse_attn_workspace_size(const csa2_attn_args* a) {
  if (!a || a->n_rows <= 0) return 0;
  return attn_workspace(a, attn_splits(a->n_rows, a->K, a->window));
}

csa2_status csa2_sparse_attn(const csa2_attn_args* a, void* stream) {
  csa2_status st = check_attn(a, true);
  if (st != CSA2_OK || a->n_rows == 0) return st;
  const size_t need = csa2_sparse_attn_workspace_size(a);
  if (need > 0 && (!a->workspace || a->workspace_bytes < need)) return CSA2_EWORKSPACE;
  return run_attn(a, a->idx, static_cast<uint8_t*>(a->workspace), static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------- fused decode layer
// Workspace: [segment lists | block maxima | kept blocks | attention partials]
static size_t decode_ws(const csa2_decode_args* a, int* n_seg_out) {
  const csa2_index_args* ix = &a->index;
  const int n_rows = a->attn.n_rows;
  size_t ws = 0;
  int n_seg = 1;
  if (a->mode != CSA2_MODE_REUSE) {
    const long long L = a->mode == CSA2_MODE_REINDEX ? a->pool_len : ix->n_records;
    csa2_index_args ic = *ix;
    ic.cand = a->mode == CSA2_MODE_REINDEX ? a->pool : nullptr;
    ic.block_max = nullptr;
    const int cand_run = a->mode == CSA2_MODE_REINDEX ? a->block_size : 0;
    const ScanPath path = scan_path(&ic, true, cand_run, a->mode == CSA2_MODE_FULL ? a->K : 0);
    if (path == ScanPath::kTc05Stream) {
      n_seg = stream_segments(n_rows, L);
    } else if (path == ScanPath::kTc05Decode) {
      const int unit = a->mode == CSA2_MODE_FULL_POOL ? a->block_size : 128;
      // segments of at least 512 records: short rows (a 2,048-record decode row: four
      // segments) stream in parallel blocks and select as a cluster (34.4 -> 29.1 us)
      n_seg = tc05_segments(n_rows, L, unit, 512);
      // A row's segments select its top-K together as one thread-block cluster of at most 16
      // blocks; where more segments were planned, 16 per row still keep at least 64 blocks
      // streaming and each segment within shared memory, and save the list merge.
      const long long units = (L + unit - 1) / unit;
      if (n_seg > 16 && (long long)n_rows * 16 >= 64 && (units + 15) / 16 <= mma_decode_max_seg_blocks() &&
          (units + 15) / 16 <= mma_decode_max_segment() / unit)
        n_seg = 16;
      // Clusters larger than 8 are resident only where the GPU's processor clusters have room
      // for all of them at once; otherwise the largest of 12 or 8 that is (the cluster
      // selection is worth more than the extra streaming blocks: 8 rows x 128 K records,
      // 16 non-resident segments against 12 resident ones: 107 -> 101 us for the layer).
      const bool fp8 = ic.k_dtype == CSA2_FP8_E4M3_ROWSCALE;
      auto seg_blocks = [&](int ns) {
        const long long per = (units + ns - 1) / ns;
        return a->mode == CSA2_MODE_FULL_POOL ? (int)per : a->mode == CSA2_MODE_REINDEX ? (int)(2 * per) : 0;
      };
      if (n_seg > 8 && tuning(CSA2_TUNE_SCAN_CLUSTER) != 0 &&
          !mma_decode_cluster_ok(n_seg, n_rows, a->K, seg_blocks(n_seg), fp8)) {
        for (const int ns : {12, 8}) {
          if (ns >= n_seg || (long long)n_rows * ns < 64) continue;
          if ((units + ns - 1) / ns > mma_decode_max_segment() / unit) continue;
          if (seg_blocks(ns) > mma_decode_max_seg_blocks()) continue;
          if (mma_decode_cluster_ok(ns, n_rows, a->K, seg_blocks(ns), fp8)) {
            n_seg = ns;
            break;
          }
        }
      }
    } else {  // candidate lists (Reindex) are short: smaller segments keep enough blocks busy
      n_seg = scan_segments(n_rows, L, a->mode == CSA2_MODE_REINDEX ? 512 : 4096);
    }
    ws += lists_bytes(n_rows, n_seg, a->K);
    if (n_seg > 1) ws += align_up((size_t)n_rows * 8);  // per-row completion counters
    if (a->mode == CSA2_MODE_FULL_POOL) {
      const long long nb = (ix->n_records + a->block_size - 1) / a->block_size;
      ws += align_up((size_t)n_rows * nb * 4) + align_up((size_t)n_rows * a->n_keep * 4);
    }
  }
  ws += attn_workspace(&a->attn, attn_splits(n_rows, a->K, a->attn.window));
  if (n_seg_out) *n_seg_out = n_seg;
  return ws;
}

size_t csa2_fused_decode_workspace_size(const csa2_decode_args* a) {
  if (!a || a->attn.n_rows <= 0 || a->K < 1) return 0;
  return decode_ws(a, nullptr);
}

csa2_status csa2_fused_decode(const csa2_decode_args* a, void* stream) {
  if (!a) return CSA2_EINVAL;
  if (a->mode < CSA2_MODE_FULL || a->mode > CSA2_MODE_REUSE) return CSA2_EINVAL;
  if (a->K < 1 || a->K > kScanMaxK) return CSA2_EUNSUPPORTED;
  if (!a->idx) return CSA2_EINVAL;
  csa2_attn_args at = a->attn;
  at.K = a->K;
  csa2_status st = check_attn(&at, false);
  if (st != CSA2_OK || at.n_rows == 0) return st;
  const csa2_index_args* ix = &a->index;
  if (a->mode != CSA2_MODE_REUSE) {
    csa2_index_args ic = *ix;
    ic.cand = nullptr;
    ic.scores = nullptr;
    ic.block_max = nullptr;
    st = check_index(&ic, false);
    if (st != CSA2_OK) return st;
    if (ix->n_rows != at.n_rows || ix->n_records != at.n_records) return CSA2_EINVAL;
  }
  if (a->mode == CSA2_MODE_FULL_POOL) {
    if (!pow2(a->block_size) || a->block_size < 16 || a->block_size > 4096) return CSA2_EUNSUPPORTED;
    if (a->n_keep < 1 || a->n_keep > CSA2_MAX_TOPK) return CSA2_EUNSUPPORTED;
    if (a->pool_len != a->n_keep * a->block_size || !a->pool || !a->n_pool) return CSA2_EINVAL;
  }
  if (a->mode == CSA2_MODE_REINDEX && (!a->pool || !a->n_pool || a->pool_len < 1)) return CSA2_EINVAL;
  int n_seg = 1;
  const size_t need = decode_ws(a, &n_seg);
  if (need > 0 && (!a->workspace || a->workspace_bytes < need)) return CSA2_EWORKSPACE;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int n_rows = at.n_rows;
  Carve c{static_cast<uint8_t*>(a->workspace)};
  cudaError_t e = cudaSuccess;
  auto mark = [&](int i) {
    if (a->stage_events[i]) cudaEventRecord(static_cast<cudaEvent_t>(a->stage_events[i]), s);
  };
  if (a->mode == CSA2_MODE_REUSE) {  // no indexing stages: events 0 and 1 mark the same point
    mark(0);
    mark(1);
  }
  if (a->mode != CSA2_MODE_REUSE) {
    ScanParams p = scan_params(ix);
    p.K = a->K;
    p.idx = a->idx;
    if (n_seg > 1) {
      p.seg_keys = c.take<uint32_t>((size_t)n_rows * n_seg * a->K);
      p.seg_pos = c.take<int32_t>((size_t)n_rows * n_seg * a->K);
      p.seg_cnt = c.take<int32_t>((size_t)n_rows * n_seg);
      p.seg_thr = c.take<uint32_t>((size_t)n_rows * n_seg);
    }
    int32_t* kept = nullptr;
    if (a->mode == CSA2_MODE_FULL_POOL) {
      p.n_blocks = (ix->n_records + a->block_size - 1) / a->block_size;
      p.bmax_stride = p.n_blocks;
      p.block_max = c.take<float>((size_t)n_rows * p.n_blocks);
      p.unit = a->block_size;
      kept = c.take<int32_t>((size_t)n_rows * a->n_keep);
    }
    csa2_index_args ic = *ix;
    ic.cand = nullptr;
    ic.block_max = nullptr;
    if (a->mode == CSA2_MODE_REINDEX) {
      p.cand = a->pool;
      p.n_cand = a->n_pool;
      p.cand_stride = a->pool_len;
      p.cand_run = a->block_size;
      ic.cand = a->pool;
      ic.L = a->pool_len;
    }
    const int stream_k = a->mode == CSA2_MODE_FULL ? a->K : 0;
    const ScanPath path = scan_path(&ic, true, p.cand_run, stream_k);
    const bool tc05 = path == ScanPath::kTc05Decode;
    if ((tc05 && a->mode != CSA2_MODE_FULL_POOL) || path == ScanPath::kTc05Stream) p.unit = 128;
    p.dev_status = at.dev_status;
    const int seg_blocks = p.block_max ? (int)(((ic.n_records + p.unit - 1) / p.unit + n_seg - 1) / n_seg)
                           : p.cand   ? (int)(2 * (((ic.L + p.unit - 1) / p.unit + n_seg - 1) / n_seg))
                                      : 0;
    p.cluster_merge = tc05 && tuning(CSA2_TUNE_SCAN_CLUSTER) != 0 && mma_decode_cluster_ok(n_seg, n_rows, a->K, seg_blocks, ic.k_dtype == CSA2_FP8_E4M3_ROWSCALE);
    const bool fused_merge = tc05 && !p.cluster_merge && mma_decode_can_merge(n_seg, a->K);
    if (n_seg > 1) {
      p.row_done = c.take<unsigned long long>((size_t)n_rows);
      p.call_tag = next_call_tag();
      if (!fused_merge) p.row_done = nullptr;
    }
    if (p.cluster_merge) p.seg_keys = nullptr, p.seg_pos = nullptr, p.seg_cnt = nullptr, p.seg_thr = nullptr;
    mark(0);  // stage 0: the indexer scan kernel alone
    e = launch_scan(p, &ic, true, n_seg, s, stream_k);
    if (e != cudaSuccess) return CSA2_ECUDA;
    mark(1);
    if (n_seg > 1 && !fused_merge && !p.cluster_merge) {
      FeedParams m{};
      m.n_rows = n_rows;
      m.K = a->K;
      m.in_keys = p.seg_keys;
      m.in_pos = p.seg_pos;
      m.in_cnt = p.seg_cnt;
      m.in_thr = p.seg_thr;
      m.in_seg = n_seg;
      m.in_K = a->K;
      m.idx = a->idx;
      e = launch_lists_merge(m, s);
      if (e != cudaSuccess) return CSA2_ECUDA;
    }
    if (a->mode == CSA2_MODE_FULL_POOL) {
      FeedParams f{};
      f.n_rows = n_rows;
      f.K = a->n_keep;
      f.scores = p.block_max;
      f.scores_stride = p.n_blocks;
      f.n_valid = ix->n_visible;
      f.valid_div = a->block_size;
      f.idx = kept;
      f.pool = a->pool;
      f.n_pool = a->n_pool;
      f.pool_bs = a->block_size;
      e = launch_topk_feed(f, false, 1, s);  // block selection and the pool's positions
      if (e != cudaSuccess) return CSA2_ECUDA;
    }
  }
  mark(2);
  st = run_attn(&at, a->idx, static_cast<uint8_t*>(a->workspace) + c.off, s);
  mark(3);
  return st;
}

csa2_status csa2_write_records(const csa2_write_args* a, void* stream) {
  if (!a || a->n_rows < 0) return CSA2_EINVAL;
  if (a->n_rows == 0) return CSA2_OK;
  if (!a->x || !a->dst_row || !a->codes || (!a->scales && a->out_dtype != CSA2_BF16) || a->cache_rows < 1)
    return CSA2_EINVAL;
  const bool fp8 = a->out_dtype == CSA2_FP8_E4M3_ROWSCALE, bf16 = a->out_dtype == CSA2_BF16;
  if (!fp8 && !bf16 && a->out_dtype != CSA2_FP4_E2M1_G16 && a->out_dtype != CSA2_FP4_E2M1_G32) return CSA2_EINVAL;
  if (!aligned(a->x, 16) || !aligned(a->codes, 16) || !aligned(a->dst_row, 8) || (a->pos && !aligned(a->pos, 8)) ||
      (fp8 && !aligned(a->scales, 4)))
    return CSA2_EINVAL;
  WriteParams p{};
  p.n_rows = a->n_rows;
  p.x = a->x;
  p.x_f32 = a->x_f32 != 0;
  p.pos = a->pos;
  for (int i = 0; i < CSA2_ROPE_DIM / 2; ++i)
    p.inv_freq[i] = std::pow((double)a->rope_theta, -2.0 * i / (double)CSA2_ROPE_DIM);
  p.dst_row = a->dst_row;
  p.cache_rows = a->cache_rows;
  p.out_dtype = a->out_dtype;
  p.codes = a->codes;
  p.scales = a->scales;
  p.dev_status = a->dev_status;
  return cuda_status(launch_write_records(p, static_cast<cudaStream_t>(stream)));
}

csa2_status csa2_compress(const csa2_compress_args* a, void* stream) {
  if (!a || a->n_entries < 0) return CSA2_EINVAL;
  if (a->n_entries == 0) return CSA2_OK;
  if (!a->kv || !a->gate || !a->out || a->ratio < 1 || a->ratio > 8) return CSA2_EINVAL;
  if (!aligned(a->kv, 16) || !aligned(a->gate, 16) || !aligned(a->out, 16)) return CSA2_EINVAL;
  return cuda_status(launch_compress(a->n_entries, a->ratio, a->kv, a->gate, a->x_f32 != 0, a->out,
                                     static_cast<cudaStream_t>(stream)));
}

size_t csa2_query_proj_workspace_size(const csa2_query_proj_args* a) {
  if (!a || a->n_tokens <= 0 || a->q_rank <= 0) return 0;
  return align_up((size_t)a->n_tokens * a->q_rank * 2) + align_up((size_t)(a->q_rank / 128) * 8 * a->n_tokens * 4);
}

csa2_status csa2_query_proj(const csa2_query_proj_args* a, void* stream) {
  if (!a || a->n_tokens < 0) return CSA2_EINVAL;
  if (a->n_tokens == 0) return CSA2_OK;
  if (a->hidden < 64 || a->hidden % 64 || a->q_rank < 128 || a->q_rank % 128 || a->n_heads < 1 ||
      a->n_heads > 4096 || !(a->eps >= 0.f))
    return CSA2_EINVAL;
  if (!a->x || !a->w_dq || !a->w_uq || !a->q || !aligned(a->x, 16) || !aligned(a->w_dq, 16) ||
      !aligned(a->w_uq, 16) || !aligned(a->q, 16))
    return CSA2_EINVAL;
  if (!a->workspace || !aligned(a->workspace, 16) || a->workspace_bytes < csa2_query_proj_workspace_size(a))
    return CSA2_EWORKSPACE;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int T = a->n_tokens;
  Carve c{static_cast<uint8_t*>(a->workspace)};
  uint16_t* cq = c.take<uint16_t>((size_t)T * a->q_rank);
  float* ss = c.take<float>((size_t)(a->q_rank / 128) * 8 * T);  // per feature tile and K split
  int ss_tiles = 0;
  // down-projection: c * g_q in bf16 and per-token partial sums of squares
  {
    const int m_tiles = a->q_rank / 128, k_steps = a->hidden / 64;
    const ProjPlan pl = proj_plan(T, k_steps, m_tiles * ((T + proj_bn(T) - 1) / proj_bn(T)), true);
    CUtensorMap tmA, tmB;
    if (!make_tmap_bf16(&tmA, a->w_dq, a->hidden, a->q_rank, (unsigned long long)a->hidden * 2, 128) ||
        !make_tmap_bf16(&tmB, a->x, a->hidden, T, (unsigned long long)a->hidden * 2, pl.bn))
      return CSA2_ECUDA;
    ProjParams p{};
    p.mode = kProjDown;
    p.n_tok = T;
    p.k_steps = k_steps;
    p.m_tiles = m_tiles;
    p.ks = pl.ks;
    p.bn = pl.bn;
    p.stages = pl.stages;
    p.out = cq;
    p.out_ld = a->q_rank;
    p.gain = a->g_q;
    p.ss = ss;
    p.dev_status = a->dev_status;
    ss_tiles = m_tiles * pl.ks;
    const cudaError_t e = launch_proj(tmA, tmB, p, 1, s);
    if (e != cudaSuccess) return CSA2_ECUDA;
  }
  // up-projection with the RMSNorm factors and the per-head RMSNorm
  {
    const int m_tiles = a->n_heads * (CSA2_HEAD_DIM / 128), k_steps = a->q_rank / 64;
    const ProjPlan pl = proj_plan(T, k_steps, m_tiles * ((T + proj_bn(T) - 1) / proj_bn(T)), false);
    CUtensorMap tmA, tmB;
    if (!make_tmap_bf16(&tmA, a->w_uq, a->q_rank, (unsigned long long)a->n_heads * CSA2_HEAD_DIM,
                        (unsigned long long)a->q_rank * 2, 128) ||
        !make_tmap_bf16(&tmB, cq, a->q_rank, T, (unsigned long long)a->q_rank * 2, pl.bn))
      return CSA2_ECUDA;
    ProjParams p{};
    p.mode = kProjUp;
    p.n_tok = T;
    p.k_steps = k_steps;
    p.m_tiles = m_tiles;
    p.ks = 1;
    p.bn = pl.bn;
    p.stages = pl.stages;
    p.out = a->q;
    p.out_ld = (long long)a->n_heads * CSA2_HEAD_DIM;
    p.gain = a->g_head;
    p.ss = ss;
    p.ss_tiles = ss_tiles;
    p.inv_rank = 1.f / (float)a->q_rank;
    p.eps = a->eps;
    p.dev_status = a->dev_status;
    const cudaError_t e = launch_proj(tmA, tmB, p, 1, s);
    if (e != cudaSuccess) return CSA2_ECUDA;
  }
  return CSA2_OK;
}

size_t csa2_out_proj_workspace_size(const csa2_out_proj_args* a) {
  if (!a || a->n_tokens <= 0 || a->n_groups <= 0 || a->o_rank <= 0) return 0;
  return align_up((size_t)a->n_tokens * a->n_groups * a->o_rank * 2);
}

csa2_status csa2_out_proj(const csa2_out_proj_args* a, void* stream) {
  if (!a || a->n_tokens < 0) return CSA2_EINVAL;
  if (a->n_tokens == 0) return CSA2_OK;
  if (a->n_groups < 1 || a->n_heads < a->n_groups || a->n_heads % a->n_groups || a->n_heads > 4096 ||
      a->o_rank < 128 || a->o_rank % 128 || a->hidden < 128 || a->hidden % 128)
    return CSA2_EINVAL;
  if (!a->o || !a->w_oa || !a->w_ob || !a->out || !aligned(a->o, 16) || !aligned(a->w_oa, 16) ||
      !aligned(a->w_ob, 16) || !aligned(a->out, 16))
    return CSA2_EINVAL;
  if (!a->workspace || !aligned(a->workspace, 16) || a->workspace_bytes < csa2_out_proj_workspace_size(a))
    return CSA2_EWORKSPACE;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int T = a->n_tokens, G = a->n_groups;
  const long long kg = (long long)a->n_heads / G * CSA2_HEAD_DIM, cols = (long long)a->n_heads * CSA2_HEAD_DIM;
  const long long yr = (long long)G * a->o_rank;
  uint16_t* y = static_cast<uint16_t*>(a->workspace);
  // per group: y_g = W_OA[g] o_g
  {
    const int m_tiles = a->o_rank / 128, k_steps = (int)(kg / 64);
    const ProjPlan pl = proj_plan(T, k_steps, m_tiles * G * ((T + proj_bn(T) - 1) / proj_bn(T)), true);
    CUtensorMap tmA, tmB;
    if (!make_tmap_bf16(&tmA, a->w_oa, kg, (unsigned long long)yr, (unsigned long long)kg * 2, 128) ||
        !make_tmap_bf16(&tmB, a->o, cols, T, (unsigned long long)cols * 2, pl.bn))
      return CSA2_ECUDA;
    ProjParams p{};
    p.mode = kProjPlain;
    p.n_tok = T;
    p.k_steps = k_steps;
    p.m_tiles = m_tiles;
    p.ks = pl.ks;
    p.bn = pl.bn;
    p.stages = pl.stages;
    p.a_rows_per_group = a->o_rank;
    p.b_cols_per_group = (int)kg;
    p.out = y;
    p.out_ld = yr;
    p.out_cols_per_group = a->o_rank;
    p.dev_status = a->dev_status;
    if (launch_proj(tmA, tmB, p, G, s) != cudaSuccess) return CSA2_ECUDA;
  }
  // out = W_OB y
  {
    const int m_tiles = a->hidden / 128, k_steps = (int)(yr / 64);
    const ProjPlan pl = proj_plan(T, k_steps, m_tiles * ((T + proj_bn(T) - 1) / proj_bn(T)), true);
    CUtensorMap tmA, tmB;
    if (!make_tmap_bf16(&tmA, a->w_ob, yr, a->hidden, (unsigned long long)yr * 2, 128) ||
        !make_tmap_bf16(&tmB, y, yr, T, (unsigned long long)yr * 2, pl.bn))
      return CSA2_ECUDA;
    ProjParams p{};
    p.mode = kProjPlain;
    p.n_tok = T;
    p.k_steps = k_steps;
    p.m_tiles = m_tiles;
    p.ks = pl.ks;
    p.bn = pl.bn;
    p.stages = pl.stages;
    p.out = a->out;
    p.out_ld = a->hidden;
    p.dev_status = a->dev_status;
    if (launch_proj(tmA, tmB, p, 1, s) != cudaSuccess) return CSA2_ECUDA;
  }
  return CSA2_OK;
}

csa2_status csa2_expand_mxfp4(const csa2_expand_args* a, void* stream) {
  if (!a || a->n_records < 0) return CSA2_EINVAL;
  if (a->n_records == 0) return CSA2_OK;
  if (!a->codes || !a->exps || !a->out || !aligned(a->codes, 16) || !aligned(a->out, 16)) return CSA2_EINVAL;
  return cuda_status(
      launch_expand_mxfp4(a->n_records, a->codes, a->exps, a->out, static_cast<cudaStream_t>(stream)));
}

csa2_status csa2_linear(const csa2_linear_args* a, void* stream) {
  if (!a || a->n_tokens < 0) return CSA2_EINVAL;
  if (a->n_tokens == 0) return CSA2_OK;
  if (a->in_features < 64 || a->in_features % 64 || a->out_features < 128 || a->out_features % 128)
    return CSA2_EINVAL;
  if (!a->x || !a->w || !a->out || !aligned(a->x, 16) || !aligned(a->w, 16) || !aligned(a->out, 16))
    return CSA2_EINVAL;
  const int T = a->n_tokens, m_tiles = a->out_features / 128, k_steps = a->in_features / 64;
  const ProjPlan pl = proj_plan(T, k_steps, m_tiles * ((T + proj_bn(T) - 1) / proj_bn(T)), true);
  CUtensorMap tmA, tmB;
  if (!make_tmap_bf16(&tmA, a->w, a->in_features, a->out_features, (unsigned long long)a->in_features * 2, 128) ||
      !make_tmap_bf16(&tmB, a->x, a->in_features, T, (unsigned long long)a->in_features * 2, pl.bn))
    return CSA2_ECUDA;
  ProjParams p{};
  p.mode = kProjPlain;
  p.n_tok = T;
  p.k_steps = k_steps;
  p.m_tiles = m_tiles;
  p.ks = pl.ks;
  p.bn = pl.bn;
  p.stages = pl.stages;
  p.out = a->out;
  p.out_ld = a->out_features;
  p.dev_status = a->dev_status;
  return cuda_status(launch_proj(tmA, tmB, p, 1, static_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------------- record-range split
size_t csa2_shard_candidates_workspace_size(const csa2_shard_args* a) {
  if (!a || a->n_rows <= 0 || a->K < 1) return 0;
  csa2_topk_args t{};
  t.n_rows = a->n_rows;
  t.L = a->L;
  t.K = a->K;
  return csa2_topk_workspace_size(&t);
}

csa2_status csa2_shard_candidates(const csa2_shard_args* a, void* stream) {
  if (!a || a->n_rows < 0) return CSA2_EINVAL;
  if (a->n_rows == 0) return CSA2_OK;
  if (!a->scores || !a->n_valid || !a->out_scores || !a->out_pos || !a->out_cnt || a->first_record < 0 ||
      a->L < 1 || a->L > (1LL << 24) || a->first_record + a->L > (1LL << 31) - 1)
    return CSA2_EINVAL;
  if (a->K < 1 || a->K > CSA2_MAX_TOPK) return CSA2_EUNSUPPORTED;
  // the range's exact top-K columns (into out_pos), then their scores and record positions
  csa2_topk_args t{};
  t.scores = a->scores;
  t.n_valid = a->n_valid;
  t.n_rows = a->n_rows;
  t.L = a->L;
  t.K = a->K;
  t.idx = a->out_pos;
  t.workspace = a->workspace;
  t.workspace_bytes = a->workspace_bytes;
  const csa2_status st = csa2_topk(&t, stream);
  if (st != CSA2_OK) return st;
  return cuda_status(launch_shard_list(a->n_rows, a->K, a->out_pos, a->scores, a->L, a->first_record, a->out_scores,
                                       a->out_pos, a->out_cnt, static_cast<cudaStream_t>(stream)));
}

size_t csa2_merge_candidates_workspace_size(const csa2_merge_args* a) {
  if (!a || a->n_rows <= 0 || a->n_lists < 1 || a->K_in < 1) return 0;
  return 2 * align_up((size_t)a->n_rows * a->n_lists * a->K_in * 4) + align_up((size_t)a->n_rows * a->n_lists * 4);
}

csa2_status csa2_merge_candidates(const csa2_merge_args* a, void* stream) {
  if (!a || a->n_rows < 0) return CSA2_EINVAL;
  if (a->n_rows == 0) return CSA2_OK;
  if (!a->scores || !a->pos || !a->cnt || !a->idx || a->n_lists < 1 || a->K_in < 1) return CSA2_EINVAL;
  if (a->n_lists > 64 || a->K_in > CSA2_MAX_TOPK || a->K < 1 || a->K > CSA2_MAX_TOPK) return CSA2_EUNSUPPORTED;
  const size_t need = csa2_merge_candidates_workspace_size(a);
  if (!a->workspace || a->workspace_bytes < need || !aligned(a->workspace, 16)) return CSA2_EWORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Carve c{static_cast<uint8_t*>(a->workspace)};
  uint32_t* keys = c.take<uint32_t>((size_t)a->n_rows * a->n_lists * a->K_in);
  int32_t* pos = c.take<int32_t>((size_t)a->n_rows * a->n_lists * a->K_in);
  int32_t* cnt = c.take<int32_t>((size_t)a->n_rows * a->n_lists);
  if (launch_lists_to_rows(a->n_rows, a->n_lists, a->K_in, a->scores, a->pos, a->cnt, keys, pos, cnt, s) != cudaSuccess)
    return CSA2_ECUDA;
  FeedParams m{};
  m.n_rows = a->n_rows;
  m.K = a->K;
  m.in_keys = keys;
  m.in_pos = pos;
  m.in_cnt = cnt;
  m.in_thr = nullptr;
  m.in_seg = a->n_lists;
  m.in_K = a->K_in;
  m.idx = a->idx;
  return cuda_status(launch_lists_merge(m, s));
}

int32_t csa2_attn_partial_tiles(int32_t K, int32_t window) {
  if (K < 0 || window < 0 || K + window < 1) return 0;
  return (K + window + 127) / 128;
}

csa2_status csa2_sparse_attn_partial(const csa2_partial_args* a, void* stream) {
  if (!a) return CSA2_EINVAL;
  const csa2_status st = check_attn(&a->attn, true, false);
  if (st != CSA2_OK || a->attn.n_rows == 0) return st;
  if (!a->part_o || !a->part_ml || !aligned(a->part_o, 16) || !aligned(a->part_ml, 8)) return CSA2_EINVAL;
  if (a->range_count < 0 || a->range_first < 0 || (a->range_count > 0 && a->range_count > a->attn.n_records))
    return CSA2_EINVAL;
  AttnParams p = attn_params(&a->attn, a->attn.idx);
  p.part_o = a->part_o;
  p.part_ml = a->part_ml;
  p.range_first = a->range_first;
  p.range_count = a->range_count;
  p.skip_window = a->skip_window != 0;
  return cuda_status(launch_attn_tiles(p, csa2_attn_partial_tiles(a->attn.K, a->attn.window),
                                       static_cast<cudaStream_t>(stream)));
}

csa2_status csa2_attn_merge(const csa2_attn_merge_args* a, void* stream) {
  if (!a || a->n_rows < 0) return CSA2_EINVAL;
  if (a->n_rows == 0) return CSA2_OK;
  if (!a->part_o || !a->part_ml || !a->q_pos || !a->sink || !a->out || a->n_parts < 1 || a->part_tiles < 1 ||
      !aligned(a->part_o, 16) || !aligned(a->part_ml, 8) || !aligned(a->out, 16) || !(a->rope_theta > 0.f))
    return CSA2_EINVAL;
  if ((long long)a->n_parts * a->part_tiles > 32) return CSA2_EUNSUPPORTED;
  AttnParams p{};
  p.n_rows = a->n_rows;
  p.q_pos = a->q_pos;
  p.sink = a->sink;
  for (int i = 0; i < CSA2_ROPE_DIM / 2; ++i)
    p.inv_freq[i] = std::pow((double)a->rope_theta, -2.0 * i / (double)CSA2_ROPE_DIM);
  p.part_o = const_cast<float*>(a->part_o);
  p.part_ml = const_cast<float*>(a->part_ml);
  p.part_tiles = a->part_tiles;
  p.part_stride_o = (long long)a->n_rows * a->part_tiles * CSA2_HEADS * CSA2_HEAD_DIM;
  p.part_stride_ml = (long long)a->n_rows * a->part_tiles * CSA2_HEADS * 2;
  p.out = a->out;
  p.out_bf16 = a->out_bf16 != 0;
  p.sink_mass = a->sink_mass;
  return cuda_status(launch_attn_merge(p, a->n_parts * a->part_tiles, static_cast<cudaStream_t>(stream)));
}

int32_t csa2_fused_decode_launch_count(const csa2_decode_args* a) {
  if (!a || a->attn.n_rows <= 0) return 0;
  int n_seg = 1;
  decode_ws(a, &n_seg);
  int n = 0;
  if (a->mode != CSA2_MODE_REUSE) {
    csa2_index_args ic = a->index;
    ic.cand = a->mode == CSA2_MODE_REINDEX ? a->pool : nullptr;
    ic.block_max = nullptr;
    if (a->mode == CSA2_MODE_REINDEX) ic.L = a->pool_len;
    const bool tc05 = scan_path(&ic, true, a->mode == CSA2_MODE_REINDEX ? a->block_size : 0,
                                a->mode == CSA2_MODE_FULL ? a->K : 0) == ScanPath::kTc05Decode;
    const int unit = a->mode == CSA2_MODE_FULL_POOL ? a->block_size : 128;
    const int seg_blocks =
        a->mode == CSA2_MODE_FULL_POOL ? (int)(((ic.n_records + unit - 1) / unit + n_seg - 1) / n_seg)
        : a->mode == CSA2_MODE_REINDEX ? (int)(2 * (((ic.L + unit - 1) / unit + n_seg - 1) / n_seg))
                                       : 0;
    const bool merged = tc05 && ((tuning(CSA2_TUNE_SCAN_CLUSTER) != 0 &&
                                  mma_decode_cluster_ok(n_seg, a->attn.n_rows, a->K, seg_blocks, ic.k_dtype == CSA2_FP8_E4M3_ROWSCALE)) ||
                                 mma_decode_can_merge(n_seg, a->K));
    n += 1 + (n_seg > 1 && !merged ? 1 : 0);  // the tcgen05 scan merges its segments itself
    if (a->mode == CSA2_MODE_FULL_POOL) n += 1;  // block selection writing the pool
  }
  n += 2;  // attention tiles and their merge
  return n;
}

}  // extern "C"
