// Exact top-K of materialised rows and the merge of per-segment lists (the streaming
// engine of select.cuh fed from global memory), and the expansion of kept blocks into the
// hierarchical candidate pool ("DeepSeek-V4.1-Flash explained", section 3: a block is
// scored by its best position and every position of a kept block enters the pool).
#include "select.cuh"
#include "kernels.h"

namespace csa2 {

namespace {

constexpr int kFeedWarps = 16;
constexpr int kFeedThreads = kFeedWarps * 32;

// One thread block per (output segment, row).  Entries of the row are a flat stream split
// into contiguous ranges: output segments, then warps; each warp feeds 128 entries per round.
// Source A (scores): entry j = column j, its position cand[row, j] (or j).  Source B (lists
// of earlier segments): the entries are the lists' (key, position) pairs and the position
// itself orders them.
template <bool FROM_LISTS>
__global__ void __launch_bounds__(kFeedThreads, 1) topk_feed_kernel(const FeedParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  Engine<kFeedWarps> e;
  e.sh = reinterpret_cast<EngShared*>(smem);
  e.cap = p.K + kRoundEntries;
  e.keys = reinterpret_cast<uint32_t*>(smem + sizeof(EngShared));
  e.js = reinterpret_cast<int32_t*>(e.keys + kFeedWarps * e.cap);
  e.out_key = reinterpret_cast<uint32_t*>(e.js + kFeedWarps * e.cap);
  e.out_j = reinterpret_cast<int32_t*>(e.out_key + p.K);
  e.bar_id = 0;
  e.tid = threadIdx.x;
  const int wid = threadIdx.x >> 5;
  const int row = blockIdx.y, seg = blockIdx.x, n_seg = gridDim.x;

  const long long total = FROM_LISTS ? (long long)p.in_seg * p.in_K
                                      : ((long long)p.n_valid[row] + p.valid_div - 1) / p.valid_div;
  long long s0, s1, w0, w1;
  split_range(total, n_seg, seg, s0, s1);
  split_range(s1 - s0, kFeedWarps, wid, w0, w1);
  const long long f0 = s0 + w0, f1 = s0 + w1;
  const long long per_warp_max = ((s1 - s0) + kFeedWarps - 1) / kFeedWarps;
  const int rounds = (int)((per_warp_max + kRoundEntries - 1) / kRoundEntries);

  // Lists of earlier segments: the row's K-th key is at least the K-th key of every full
  // list, so any entry below the largest of those cannot be selected.
  uint32_t thr0 = 0u;
  if (FROM_LISTS && p.in_thr != nullptr)
    for (int s = 0; s < p.in_seg; ++s) thr0 = max(thr0, p.in_thr[(size_t)row * p.in_seg + s]);
  eng_init(e, thr0);
  int cnt = 0;
  uint32_t thr = thr0;
  constexpr int G = kRoundEntries / 32;
  long long f = f0 + e.lane();
  for (int r = 0; r < rounds; ++r) {
    // all loads of the round first, then the appends
    bool valid[G];
    uint32_t key[G];
    int32_t j[G];
#pragma unroll
    for (int k = 0; k < G; ++k) {
      const long long fk = f + 32 * k;
      valid[k] = fk < f1;
      key[k] = 0u;
      j[k] = 0;
      if (valid[k]) {
        if (FROM_LISTS) {
          const long long s = fk / p.in_K, i = fk % p.in_K;
          valid[k] = i < __ldg(p.in_cnt + (size_t)row * p.in_seg + s);
          const size_t o = ((size_t)row * p.in_seg + s) * p.in_K + i;
          if (valid[k]) {
            key[k] = __ldg(p.in_keys + o);
            j[k] = __ldg(p.in_pos + o);
          }
        } else {
          key[k] = score_key(__ldg(p.scores + (size_t)row * p.scores_stride + fk));
          j[k] = (int32_t)fk;
        }
      }
    }
#pragma unroll
    for (int k = 0; k < G; ++k) eng_append(e, cnt, thr, valid[k], key[k], j[k]);
    f += kRoundEntries;
    thr = eng_check(e, p.K, cnt);
  }
  uint32_t* thr_out = (n_seg > 1 && p.out_thr) ? p.out_thr + (size_t)row * n_seg + seg : nullptr;
  const int n = eng_finish(e, p.K, cnt, thr_out);
  auto position = [&](int32_t j) -> int32_t {
    if (!FROM_LISTS && p.cand != nullptr) return p.cand[(size_t)row * p.cand_stride + j];
    return j;
  };
  if (n_seg == 1) {
    int32_t* out = p.idx + (size_t)row * p.K;
    for (int i = threadIdx.x; i < p.K; i += kFeedThreads) out[i] = i < n ? position(e.out_j[i]) : -1;
  } else {
    const size_t o = ((size_t)row * n_seg + seg) * p.K;
    for (int i = threadIdx.x; i < n; i += kFeedThreads) {
      p.out_keys[o + i] = e.out_key[i];
      p.out_pos[o + i] = position(e.out_j[i]);
    }
    if (threadIdx.x == 0) p.out_cnt[(size_t)row * n_seg + seg] = n;
  }
}

// kept[row] = ascending kept block ids (-1 padded).  Only the block holding the last visible
// position can be partial, and it has the largest id of all blocks, so the visible positions
// of the kept blocks form a prefix of the pool.
__global__ void pool_expand_kernel(const int32_t* __restrict__ kept, const int32_t* __restrict__ n_visible,
                                   int n_keep, int bs, int32_t* __restrict__ pool, int32_t* __restrict__ n_pool) {
  const int row = blockIdx.x;
  const long long nv = n_visible[row];
  const int32_t* kr = kept + (size_t)row * n_keep;
  int32_t* pr = pool + (size_t)row * n_keep * bs;
  for (long long i = threadIdx.x; i < (long long)n_keep * bs; i += blockDim.x) {
    const int blk = kr[i / bs];
    long long pos = blk >= 0 ? (long long)blk * bs + i % bs : -1;
    if (pos >= nv) pos = -1;
    pr[i] = (int32_t)pos;
  }
  if (threadIdx.x == 0) {
    int nk = 0;
    while (nk < n_keep && kr[nk] >= 0) ++nk;
    long long n = 0;
    if (nk > 0) {
      const long long last = kr[nk - 1];
      n = (long long)(nk - 1) * bs + min((long long)bs, nv - last * bs);
    }
    n_pool[row] = (int32_t)n;
  }
}

}  // namespace

size_t feed_smem_bytes(int K) {
  return sizeof(EngShared) + (size_t)kFeedWarps * (K + kRoundEntries) * 8 + (size_t)K * 8;
}

cudaError_t launch_topk_feed(const FeedParams& p, bool from_lists, int out_seg, cudaStream_t stream) {
  if (p.n_rows == 0) return cudaSuccess;
  const size_t smem = feed_smem_bytes(p.K);
  dim3 grid(out_seg, p.n_rows), block(kFeedThreads);
  cudaError_t e;
  if (from_lists) {
    e = cudaFuncSetAttribute(topk_feed_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    topk_feed_kernel<true><<<grid, block, smem, stream>>>(p);
  } else {
    e = cudaFuncSetAttribute(topk_feed_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    topk_feed_kernel<false><<<grid, block, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_pool_expand(const int32_t* kept, const int32_t* n_visible, int n_rows, int n_keep,
                               int block_size, int32_t* pool, int32_t* n_pool, cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  pool_expand_kernel<<<n_rows, 256, 0, stream>>>(kept, n_visible, n_keep, block_size, pool, n_pool);
  return cudaGetLastError();
}

}  // namespace csa2
