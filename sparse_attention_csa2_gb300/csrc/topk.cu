// Exact top-K of materialised rows and the merge of per-segment lists (the streaming
// engine of select.cuh fed from global memory), and the expansion of kept blocks into the
// hierarchical candidate pool ("DeepSeek-V4.1-Flash explained", section 3: a block is
// scored by its best position and every position of a kept block enters the pool).
#include "select.cuh"
#include "kernels.h"

namespace csa2 {

namespace {

// One thread block per (output segment, row).  Entries of the row are a flat stream split
// into contiguous ranges: output segments, then warps; each warp feeds 128 entries per round.
template <bool FROM_LISTS>
__global__ void __launch_bounds__(kSelThreads, 1) topk_feed_kernel(const FeedParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  SelectShared* sh = reinterpret_cast<SelectShared*>(smem);
  TopkEngine eng;
  eng.cap = p.K + kRoundEntries;
  eng.keys = reinterpret_cast<uint32_t*>(smem + sizeof(SelectShared));
  eng.pos = reinterpret_cast<int32_t*>(eng.keys + kSelWarps * eng.cap);
  eng.sh = sh;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int row = blockIdx.y, seg = blockIdx.x, n_seg = gridDim.x;

  const long long total = FROM_LISTS ? (long long)p.in_seg * p.in_K
                                      : ((long long)p.n_valid[row] + p.valid_div - 1) / p.valid_div;
  long long s0, s1, w0, w1;
  split_range(total, n_seg, seg, s0, s1);
  split_range(s1 - s0, kSelWarps, wid, w0, w1);
  const long long f0 = s0 + w0, f1 = s0 + w1;
  const long long per_warp_max = ((s1 - s0) + kSelWarps - 1) / kSelWarps;
  const int rounds = (int)((per_warp_max + kRoundEntries - 1) / kRoundEntries);

  engine_init(eng);
  int cnt = 0;
  uint32_t thr = 0u;
  long long f = f0 + lane;
  for (int r = 0; r < rounds; ++r) {
#pragma unroll
    for (int k = 0; k < kRoundEntries / 32; ++k, f += 32) {
      bool valid = f < f1;
      uint32_t key = 0u;
      int32_t pos = 0;
      if (valid) {
        if (FROM_LISTS) {
          const long long s = f / p.in_K, i = f % p.in_K;
          valid = i < p.in_cnt[(size_t)row * p.in_seg + s];
          if (valid) {
            const size_t o = ((size_t)row * p.in_seg + s) * p.in_K + i;
            key = p.in_keys[o];
            pos = p.in_pos[o];
          }
        } else {
          key = score_key(p.scores[(size_t)row * p.scores_stride + f]);
          pos = p.cand ? p.cand[(size_t)row * p.cand_stride + f] : (int32_t)f;
        }
      }
      warp_append(eng, wid, cnt, thr, valid, key, pos);
    }
    thr = engine_round_end(eng, p.K, wid, lane, cnt);
  }
  if (n_seg == 1) {
    engine_finish(eng, p.K, wid, lane, cnt, p.idx + (size_t)row * p.K, nullptr, nullptr, nullptr);
  } else {
    const size_t o = ((size_t)row * n_seg + seg) * p.K;
    engine_finish(eng, p.K, wid, lane, cnt, nullptr, p.out_keys + o, p.out_pos + o,
                  p.out_cnt + (size_t)row * n_seg + seg);
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

size_t feed_smem_bytes(int K) { return sizeof(SelectShared) + (size_t)kSelWarps * (K + kRoundEntries) * 8; }

cudaError_t launch_topk_feed(const FeedParams& p, bool from_lists, int out_seg, cudaStream_t stream) {
  if (p.n_rows == 0) return cudaSuccess;
  const size_t smem = feed_smem_bytes(p.K);
  dim3 grid(out_seg, p.n_rows), block(kSelThreads);
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
