// Exact top-K of materialised rows and the merge of per-segment lists (the streaming
// engine of select.cuh fed from global memory), and the expansion of kept blocks into the
// hierarchical candidate pool ("DeepSeek-V4.1-Flash explained", section 3: a block is
// scored by its best position and every position of a kept block enters the pool).
#include <algorithm>

#include "array_topk.cuh"
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
    if (p.idx) {
      int32_t* out = p.idx + (size_t)row * p.K;
      for (int i = threadIdx.x; i < p.K; i += kFeedThreads) out[i] = i < n ? position(e.out_j[i]) : -1;
    }
    if (!FROM_LISTS && p.pool) {
      // Kept blocks, ascending, to their positions.  Only the block holding the last visible
      // position can be partial, and it has the largest id of all blocks, so the visible
      // positions of the kept blocks form a prefix of the pool.
      const int bs = p.pool_bs;
      const long long nv = p.n_valid[row];
      int32_t* pr = p.pool + (size_t)row * p.K * bs;
      for (long long i = threadIdx.x; i < (long long)p.K * bs; i += kFeedThreads) {
        const int r = (int)(i / bs);
        const long long blk = r < n ? position(e.out_j[r]) : -1;
        long long pos = blk >= 0 ? blk * bs + i % bs : -1;
        if (pos >= nv) pos = -1;
        pr[i] = (int32_t)pos;
      }
      if (threadIdx.x == 0) {
        long long np = 0;
        if (n > 0) np = (long long)(n - 1) * bs + min((long long)bs, nv - (long long)position(e.out_j[n - 1]) * bs);
        p.n_pool[row] = (int32_t)np;
      }
    }
  } else {
    const size_t o = ((size_t)row * n_seg + seg) * p.K;
    for (int i = threadIdx.x; i < n; i += kFeedThreads) {
      p.out_keys[o + i] = e.out_key[i];
      p.out_pos[o + i] = position(e.out_j[i]);
    }
    if (threadIdx.x == 0) p.out_cnt[(size_t)row * n_seg + seg] = n;
  }
}

// Merge of per-segment lists (source B) into a row's final top-K.  A row's lists are spread
// over a thread-block cluster (up to 8 blocks, each a contiguous range of segments, so block
// order followed by slot order is position order).  Each block stages its lists' keys in
// shared memory, keys below the largest per-segment K-th key zeroed (that segment alone holds
// K entries at or above it).  The candidates are a row's best keys and share their leading
// bits: the blocks exchange their smallest and largest candidate, and every key is shifted
// left past the bits all candidates share (bit 0 set so that no candidate becomes 0; order
// and ties are unchanged), so the histogram levels of the cluster selection spread the
// candidates instead of piling them onto a few counters.  The cluster then selects the K best
// exactly as the indexer scan's cluster does, and each block writes its share of the row's
// positions at its offset.
constexpr int kMergeWarps = 12;
constexpr int kMergeThreads = kMergeWarps * 32;
constexpr int kMergeMaxCta = 8;
constexpr int kMergeMaxLists = 128;  // lists (segments) per row

struct MergeShared {
  int cnt[kMergeMaxLists];
  uint32_t thr[kMergeMaxLists];
  uint32_t kext[2 + 2 * kMergeMaxCta];  // this block's extremes; block 0: every block's
};

__global__ void __launch_bounds__(kMergeThreads, 1) lists_merge_kernel(const FeedParams p, int seg_per_cta) {
  extern __shared__ __align__(16) uint8_t msm[];
  __shared__ ArrSelShared sh;
  __shared__ MergeShared ms;
  const int row = blockIdx.y, S = p.in_seg, Kin = p.in_K, K = p.K;
  const uint32_t rank = cluster_rank(), n_cta = gridDim.x;
  const int sg0 = min(S, (int)rank * seg_per_cta), sg1 = min(S, sg0 + seg_per_cta);
  const int n_here = (sg1 - sg0) * Kin, cap = seg_per_cta * Kin;
  // every region starts on a 16-byte boundary (the lists' room takes 16-byte stores)
  uint32_t* keys = reinterpret_cast<uint32_t*>(msm);                    // [cap, padded to 4]
  int32_t* sel_idx = reinterpret_cast<int32_t*>(keys + ((cap + 3) & ~3));  // [K, padded to 4]
  ArrSel<kMergeWarps> s;
  s.sh = &sh;
  s.tid = threadIdx.x;
  s.scratch = reinterpret_cast<uint32_t*>(sel_idx + ((K + 3) & ~3));  // lists, 16-byte aligned
  const int ln = s.lane();
  // Programmatic dependent launch: the next kernel (the attention, whose tiles over the window
  // need no indices) may start while the row selections run; it waits for this grid before it
  // reads them.  The lists are the previous kernel's output: wait for it first.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  for (int i = s.tid; i < S; i += kMergeThreads) {
    ms.cnt[i] = min(__ldcg(p.in_cnt + (size_t)row * S + i), Kin);
    ms.thr[i] = p.in_thr ? __ldcg(p.in_thr + (size_t)row * S + i) : 0u;
  }
  if (s.tid < 2) ms.kext[s.tid] = s.tid == 0 ? 0xffffffffu : 0u;
  s.zero_hist(kHistBins);
  s.sync();
  uint32_t thr0 = 0u;
  for (int i = 0; i < S; ++i) thr0 = max(thr0, ms.thr[i]);
  const uint32_t* gk = p.in_keys + ((size_t)row * S + sg0) * Kin;
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  auto stage = [&](uint32_t key, int i) -> uint32_t {
    const int sg = sg0 + i / Kin, j = i - (sg - sg0) * Kin;
    key = (j < ms.cnt[sg] && key >= thr0) ? key : 0u;
    if (key) kmin = min(kmin, key), kmax = max(kmax, key);
    return key;
  };
  if ((Kin & 3) == 0) {  // the lists' rows are 16-byte aligned
    const uint4* g4 = reinterpret_cast<const uint4*>(gk);
#pragma unroll 2
    for (int i = s.tid; i < n_here / 4; i += kMergeThreads) {
      uint4 v = __ldcg(g4 + i);
      v.x = stage(v.x, 4 * i), v.y = stage(v.y, 4 * i + 1), v.z = stage(v.z, 4 * i + 2), v.w = stage(v.w, 4 * i + 3);
      reinterpret_cast<uint4*>(keys)[i] = v;
    }
  } else {
#pragma unroll 4
    for (int i = s.tid; i < n_here; i += kMergeThreads) keys[i] = stage(__ldcg(gk + i), i);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if (ln == 0 && kmax != 0u) atomicMin(&ms.kext[0], kmin), atomicMax(&ms.kext[1], kmax);
  s.sync();
  // every block's extremes into block 0, then every block reads them all
  if (s.tid < 2) cluster_st_s32(cluster_map(&ms.kext[2 + 2 * rank + s.tid], 0), (int)ms.kext[s.tid]);
  cluster_sync();
  kmin = 0xffffffffu, kmax = 0u;
  for (uint32_t c = 0; c < n_cta; ++c) {
    const uint32_t lo = (uint32_t)cluster_ld_s32(cluster_map(&ms.kext[2 + 2 * c], 0));
    const uint32_t hi = (uint32_t)cluster_ld_s32(cluster_map(&ms.kext[3 + 2 * c], 0));
    if (hi != 0u) kmin = min(kmin, lo), kmax = max(kmax, hi);
  }
  // the bits above d are common to every candidate: shift them out
  const int d = kmax > kmin ? 31 - __clz(kmin ^ kmax) : 0;
  const int shl = kmax != 0u ? 31 - d : 0;
  for (int i = s.tid; i < n_here; i += kMergeThreads) {
    uint32_t key = keys[i];
    if (key != 0u && shl > 0) key = (key << shl) | 1u;
    keys[i] = key;
    if (key != 0u) atomicAdd(&sh.hist[key >> 20], 1);
  }
  s.sync();
  arr_threshold_impl(s, keys, n_here, K, true, ClusterPick<kMergeWarps>{rank, n_cta, cap});
  int base = 0, total = 0, kept = 0;
  if (sh.thr == 0u) {
    kept = arr_compact_cluster(s, n_here, sel_idx, rank, n_cta, &base, &total);
  } else {
    base = (int)sh.aux[2];
    total = (int)sh.aux[4];
    kept = arr_compact(s, n_here, sel_idx);
  }
  const int32_t* pos = p.in_pos + ((size_t)row * S + sg0) * Kin;
  int32_t* out = p.idx + (size_t)row * K;
  for (int r = s.tid; r < kept; r += kMergeThreads)
    if (base + r < K) out[base + r] = __ldcg(pos + sel_idx[r]);
  if (rank == n_cta - 1)
    for (int r = total + s.tid; r < K; r += kMergeThreads) out[r] = -1;
  // (the selection's last cluster barrier follows every access to another block's shared
  // memory, so the blocks may leave independently)
}

size_t merge_smem_bytes(int seg_per_cta, int Kin, int K) {
  const int cap = seg_per_cta * Kin;
  // the lists' room doubles as the cluster histogram sum (4096 words)
  return (size_t)((cap + 3) & ~3) * 4 + (size_t)((K + 3) & ~3) * 4 +
         (size_t)std::max(ArrSel<kMergeWarps>::list_words(cap), kHistBins) * 4;
}

// Exact top-K of one long row of materialised scores per block, by radix selection over the
// row held in memory (for many rows, each far longer than K: the prefill chunk's rows).
// Rows of up to 64 K entries first sample every 8th run of 128 entries for a level-1 bin g
// at or below the K-th key's (twice the proportional share of K reaches it); the level-1 pass
// also lists every entry of bin g and above, and when the K-th key's bin is at least g and the
// list held them all, the rest of the selection and the placement read only the list: about
// 1.1 passes over the row.  Otherwise, and for longer rows, pass 1 counts the keys' top 12
// bits; pass 2 counts the next 12 bits of the keys in the
// threshold's bin and lists those keys in shared memory (their number is about the bin's
// population), so the last 8 bits come from the list; when the bin holds more keys than the
// list, pass 3 counts them over the row again.  The K-th key T and the number of entries equal
// to it that are kept (the lowest positions first) then place every kept entry.  Rows of up to
// 64 K entries take one more pass, which marks the entries above T and those equal to it in two
// bitmaps (in the histogram's shared memory, free by then); the first n_eq ties in position
// order join the kept bits (a block prefix over the words' counts) and a second prefix places
// every kept entry in position order.  Longer rows take two passes: one counts each warp's kept
// entries over its contiguous range, one writes them at the warp's offset.  Loads are 16-byte
// where the row allows.
constexpr int kRtWarps = 8;
constexpr int kRtThreads = kRtWarps * 32;
constexpr int kRtList = 2048;
constexpr long long kRtBitmapMax = 65536;  // entries: two bitmaps of this many bits in `hist`

struct RowTopkShared {
  int hist[kHistBins];
  uint32_t list[kRtList];
  int32_t list_pos[kRtList];  // one-pass rows: the listed entries' indices in the row
  int n_list;
  int n_sample;
  int bin, before;
  int warp_gt[kRtWarps], warp_eq[kRtWarps];
};

// Walks entries [a, b) of the row in order, 32 per step per warp lane-contiguous; f(i, key).
template <class F>
__device__ __forceinline__ void rt_walk(const float* row, long long a, long long b, bool vec, F f) {
  const int lane = threadIdx.x & 31;
  if (vec) {
    // 128 entries per warp step, lane l: entries 4l .. 4l+3 (a is a multiple of 4 here)
    for (long long i0 = a; i0 < b; i0 += 128) {
      const long long i = i0 + 4 * lane;
      if (i + 3 < b) {
        const float4 v = *reinterpret_cast<const float4*>(row + i);
        f(i, score_key(v.x));
        f(i + 1, score_key(v.y));
        f(i + 2, score_key(v.z));
        f(i + 3, score_key(v.w));
      } else {
        for (long long k = i; k < b && k < i + 4; ++k) f(k, score_key(row[k]));
      }
    }
  } else {
    for (long long i = a + lane; i < b; i += 32) f(i, score_key(row[i]));
  }
}

// The bin (of nb, from the top) where the count from the top reaches `need`: one warp, coarse
// groups of 64 bins then the group's bins; sets sh.bin and sh.before.
__device__ __forceinline__ void rt_pick(RowTopkShared& sh, int nb, int need) {
  const int lane = threadIdx.x & 31;
  const int ng = nb / 64;  // groups (1 or 64)
  // group sums: lane l sums groups ng-1-2l and ng-2-2l (from the top)
  int g0 = 0, g1 = 0;
  const int ga = ng - 1 - 2 * lane, gb = ng - 2 - 2 * lane;
#pragma unroll 4
  for (int k = 0; k < 64; ++k) {
    if (ga >= 0) g0 += sh.hist[64 * ga + k];
    if (gb >= 0) g1 += sh.hist[64 * gb + k];
  }
  int inc = g0 + g1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  int L = __ffs(__ballot_sync(0xffffffffu, inc >= need)) - 1;
  const int acc = inc - g0 - g1;
  int grp = acc + g0 >= need ? ga : gb;
  int above = acc + g0 >= need ? acc : acc + g0;
  grp = __shfl_sync(0xffffffffu, grp, L);
  above = __shfl_sync(0xffffffffu, above, L);
  // the group's bins: lane l takes bins 63-2l and 62-2l of the group
  const int x0 = sh.hist[64 * grp + 63 - 2 * lane], x1 = sh.hist[64 * grp + 62 - 2 * lane];
  inc = x0 + x1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  L = __ffs(__ballot_sync(0xffffffffu, above + inc >= need)) - 1;
  const int acc2 = above + inc - x0 - x1;
  const int bin = acc2 + x0 >= need ? 63 - 2 * lane : 62 - 2 * lane;
  const int bef = acc2 + x0 >= need ? acc2 : acc2 + x0;
  if (lane == L) {
    sh.bin = 64 * grp + bin;
    sh.before = bef;
  }
}

// Exclusive prefix of v over the block in thread order; `total` gets the block's sum.  Uses
// sh.warp_gt as scratch (callers separate two uses by a barrier).
__device__ __forceinline__ int rt_block_scan(RowTopkShared& sh, int v, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh.warp_gt[warp] = x;
  __syncthreads();
  int before = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < kRtWarps; ++w) {
    const int c = sh.warp_gt[w];
    before += w < warp ? c : 0;
    total += c;
  }
  return before + x - v;
}

// The second half of the bitmap placement: `keep` and `tie` (in sh.hist) hold, in position
// order, the entries above T and those equal to it; the first n_eq tie bits join `keep` (a
// block prefix over the words' counts) and every kept entry is written in position order.
template <class Pos>
__device__ __forceinline__ void rt_place_marked(RowTopkShared& sh, int n_eq, long long L, int32_t* out, Pos position) {
  const int tid = threadIdx.x;
  uint32_t* keep = reinterpret_cast<uint32_t*>(sh.hist);
  uint32_t* tie = keep + kRtBitmapMax / 32;
  constexpr int kWords = (int)(kRtBitmapMax / 32), kWpt = kWords / kRtThreads;  // words per thread
  __syncthreads();
  // the first n_eq ties in position order join the kept entries (thread t: words kWpt t ..)
  const int n_words = (int)((L + 31) / 32), w0 = tid * kWpt;
  int tc = 0;
#pragma unroll
  for (int j = 0; j < kWpt; ++j) tc += w0 + j < n_words ? __popc(tie[w0 + j]) : 0;
  int total;
  int rank = rt_block_scan(sh, tc, total);
#pragma unroll
  for (int j = 0; j < kWpt; ++j) {
    if (w0 + j >= n_words) break;
    uint32_t m = tie[w0 + j], sel = 0u;
    while (m != 0u && rank < n_eq) {  // lowest bits (positions) first
      const uint32_t low = m & (0u - m);
      sel |= low;
      m ^= low;
      ++rank;
    }
    keep[w0 + j] |= sel;
  }
  __syncthreads();  // the scan's scratch is reused below
  int kc = 0;
#pragma unroll
  for (int j = 0; j < kWpt; ++j) kc += w0 + j < n_words ? __popc(keep[w0 + j]) : 0;
  int at = rt_block_scan(sh, kc, total);
#pragma unroll
  for (int j = 0; j < kWpt; ++j) {
    if (w0 + j >= n_words) break;
    uint32_t m = keep[w0 + j];
    while (m != 0u) {
      const int bit = __ffs(m) - 1;
      out[at++] = position(32LL * (w0 + j) + bit);
      m &= m - 1u;
    }
  }
}

// Placement of a row of at most kRtBitmapMax entries once the K-th key T and the number n_eq of
// entries equal to it that are kept are known: one pass over the row marks, in position order,
// the entries above T (`keep`) and equal to it (`tie`); the first n_eq tie bits join `keep`; the
// kept entries are written in position order.  Warp ranges [a, b) start on multiples of 128.
template <class Pos>
__device__ __forceinline__ void rt_place_bitmap(RowTopkShared& sh, const float* rs, long long a, long long b, bool vec,
                                                uint32_t T, int n_eq, long long L, int32_t* out, Pos position) {
  const int tid = threadIdx.x, lane = tid & 31;
  uint32_t* keep = reinterpret_cast<uint32_t*>(sh.hist);
  uint32_t* tie = keep + kRtBitmapMax / 32;
  constexpr int kWords = (int)(kRtBitmapMax / 32);
  static_assert(2 * kWords <= kHistBins, "both bitmaps fit in the histogram");
  __syncthreads();  // every thread has read the last pick's results
  for (int i = tid; i < 2 * kWords; i += kRtThreads) keep[i] = 0u;
  __syncthreads();
  if (vec) {
    for (long long i0 = a; i0 < b; i0 += 128) {
      // lane l holds entries i0 + 4l .. +3: word (i0 / 32) + l / 8, bits 4 (l % 8) .. +3
      const long long i = i0 + 4 * lane;
      float v4[4];
      if (i + 3 < b) {
        const float4 v = *reinterpret_cast<const float4*>(rs + i);
        v4[0] = v.x, v4[1] = v.y, v4[2] = v.z, v4[3] = v.w;
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) v4[u] = i + u < b ? rs[i + u] : 0.f;
      }
      uint32_t kb = 0u, tb = 0u;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const bool valid = i + u < b;
        const uint32_t key = score_key(v4[u]);
        kb |= (uint32_t)(valid && key > T) << u;
        tb |= (uint32_t)(valid && key == T) << u;
      }
      uint32_t kw = kb << (4 * (lane & 7)), tw = tb << (4 * (lane & 7));
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {
        kw |= __shfl_xor_sync(0xffffffffu, kw, o);
        tw |= __shfl_xor_sync(0xffffffffu, tw, o);
      }
      if ((lane & 7) == 0) {
        const long long wi = (i0 >> 5) + (lane >> 3);
        keep[wi] = kw;
        tie[wi] = tw;
      }
    }
  } else {
    for (long long i0 = a; i0 < b; i0 += 32) {
      const long long i = i0 + lane;
      const bool valid = i < b;
      const uint32_t key = valid ? score_key(rs[i]) : 0u;
      const uint32_t kw = __ballot_sync(0xffffffffu, valid && key > T);
      const uint32_t tw = __ballot_sync(0xffffffffu, valid && key == T);
      if (lane == 0) {
        keep[i0 >> 5] = kw;
        tie[i0 >> 5] = tw;
      }
    }
  }
  rt_place_marked(sh, n_eq, L, out, position);
}

__global__ void __launch_bounds__(kRtThreads) row_topk_kernel(const FeedParams p) {
  __shared__ RowTopkShared sh;
  const int row = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // n_valid is in [0, L] by contract; clamped so that no value reaches past the row
  const long long L = min((long long)max(p.n_valid[row], 0), p.scores_stride);
  const float* rs = p.scores + (size_t)row * p.scores_stride;
  const int K = p.K;
  int32_t* out = p.idx + (size_t)row * K;
  auto position = [&](long long j) -> int32_t {
    return p.cand != nullptr ? p.cand[(size_t)row * p.cand_stride + j] : (int32_t)j;
  };
  if (L <= K) {  // every candidate is kept
    for (int r = tid; r < K; r += kRtThreads) out[r] = r < L ? position(r) : -1;
    return;
  }
  const bool vec = ((reinterpret_cast<uintptr_t>(rs) & 15) == 0);
  // warp w's contiguous range (a multiple of 128 entries, for the 16-byte walk)
  const long long per = ((L + kRtWarps - 1) / kRtWarps + 127) / 128 * 128;
  const long long a = min(L, warp * per), b = min(L, a + per);
  // ---- one pass for rows the bitmaps cover: a sample of the row (every 8th run of 128
  // entries) gives a level-1 bin g that about twice the proportional share of K entries reach;
  // the level-1 pass then also lists every entry of bin g and above (key and index).  When the
  // K-th key's bin b1 is at least g and the list held every such entry, the two finer levels
  // and the placement come from the list; otherwise the row continues below from level 2 (the
  // level-1 histogram is complete either way).
  const bool one_pass = L <= kRtBitmapMax;
  uint32_t g = 0xffffffffu;  // no listing in the level-1 pass
  if (one_pass) {
    for (int i = tid; i < kHistBins; i += kRtThreads) sh.hist[i] = 0;
    if (tid == 0) sh.n_sample = 0;
    __syncthreads();
    const long long n_chunks = (L + 127) / 128;
    int taken = 0;
    for (long long c = 8LL * warp; c < n_chunks; c += 8LL * kRtWarps) {
      const long long c0 = c * 128, c1 = min(L, c0 + 128);
      if (vec && c0 + 4 * lane + 3 < c1) {
        const float4 v = *reinterpret_cast<const float4*>(rs + c0 + 4 * lane);
        atomicAdd(&sh.hist[score_key(v.x) >> 20], 1);
        atomicAdd(&sh.hist[score_key(v.y) >> 20], 1);
        atomicAdd(&sh.hist[score_key(v.z) >> 20], 1);
        atomicAdd(&sh.hist[score_key(v.w) >> 20], 1);
        taken += 4;
      } else {
        for (long long i = c0 + (vec ? 4 * lane : lane); i < c1 && i < c0 + (vec ? 4 * lane + 4 : 128); i += vec ? 1 : 32) {
          atomicAdd(&sh.hist[score_key(rs[i]) >> 20], 1);
          ++taken;
        }
      }
    }
    atomicAdd(&sh.n_sample, taken);
    __syncthreads();
    const int n_s = sh.n_sample;  // >= 1: the first run is sampled
    const int target = (int)min((long long)n_s, (2LL * K * n_s + L - 1) / L + 16);
    if (warp == 0) rt_pick(sh, kHistBins, target);
    __syncthreads();
    g = (uint32_t)sh.bin;
    __syncthreads();
  }
  // ---- level 1: bits 31..20 (one pass: the entries of bin g and above are also listed)
  for (int i = tid; i < kHistBins; i += kRtThreads) sh.hist[i] = 0;
  if (tid == 0) sh.n_list = 0;
  __syncthreads();
  rt_walk(rs, a, b, vec, [&](long long j, uint32_t key) {
    atomicAdd(&sh.hist[key >> 20], 1);
    if ((key >> 20) >= g) {
      const int slot = atomicAdd(&sh.n_list, 1);
      if (slot < kRtList) {
        sh.list[slot] = key;
        sh.list_pos[slot] = (int32_t)j;
      }
    }
  });
  __syncthreads();
  if (warp == 0) rt_pick(sh, kHistBins, K);
  __syncthreads();
  const uint32_t b1 = (uint32_t)sh.bin;
  int need = K - sh.before;
  const int n_listed = sh.n_list;
  __syncthreads();
  if (one_pass && b1 >= g && n_listed <= kRtList) {
    // every entry of bin b1 and above is listed
    for (int i = tid; i < kHistBins; i += kRtThreads) sh.hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n_listed; i += kRtThreads)
      if ((sh.list[i] >> 20) == b1) atomicAdd(&sh.hist[(sh.list[i] >> 8) & 0xfffu], 1);
    __syncthreads();
    if (warp == 0) rt_pick(sh, kHistBins, need);
    __syncthreads();
    const uint32_t h24 = (b1 << 12) | (uint32_t)sh.bin;
    need -= sh.before;
    __syncthreads();
    for (int i = tid; i < 256; i += kRtThreads) sh.hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n_listed; i += kRtThreads)
      if ((sh.list[i] >> 8) == h24) atomicAdd(&sh.hist[sh.list[i] & 0xffu], 1);
    __syncthreads();
    if (warp == 0) rt_pick(sh, 256, need);
    __syncthreads();
    const uint32_t T1 = (h24 << 8) | (uint32_t)sh.bin;
    const int n_eq1 = need - sh.before;
    __syncthreads();
    // the listed entries above T and equal to it, marked by position
    uint32_t* keep = reinterpret_cast<uint32_t*>(sh.hist);
    uint32_t* tie = keep + kRtBitmapMax / 32;
    for (int i = tid; i < (int)(2 * kRtBitmapMax / 32); i += kRtThreads) keep[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n_listed; i += kRtThreads) {
      const uint32_t key = sh.list[i];
      const int j = sh.list_pos[i];
      if (key > T1) atomicOr(&keep[j >> 5], 1u << (j & 31));
      else if (key == T1) atomicOr(&tie[j >> 5], 1u << (j & 31));
    }
    rt_place_marked(sh, n_eq1, L, out, position);
    return;
  }
  // ---- level 2: bits 19..8 of the keys in bin b1, which are listed on the way
  for (int i = tid; i < kHistBins; i += kRtThreads) sh.hist[i] = 0;
  if (tid == 0) sh.n_list = 0;
  __syncthreads();
  rt_walk(rs, a, b, vec, [&](long long, uint32_t key) {
    if ((key >> 20) == b1) {
      atomicAdd(&sh.hist[(key >> 8) & 0xfffu], 1);
      const int slot = atomicAdd(&sh.n_list, 1);
      if (slot < kRtList) sh.list[slot] = key;
    }
  });
  __syncthreads();
  if (warp == 0) rt_pick(sh, kHistBins, need);
  __syncthreads();
  const uint32_t hi24 = (b1 << 12) | (uint32_t)sh.bin;
  need -= sh.before;
  const int n_list = sh.n_list;
  __syncthreads();
  // ---- level 3: bits 7..0 of the keys in (b1, b2): from the list, or the row again
  for (int i = tid; i < 256; i += kRtThreads) sh.hist[i] = 0;
  __syncthreads();
  if (n_list <= kRtList) {
    for (int i = tid; i < n_list; i += kRtThreads)
      if ((sh.list[i] >> 8) == hi24) atomicAdd(&sh.hist[sh.list[i] & 0xffu], 1);
  } else {
    rt_walk(rs, a, b, vec, [&](long long, uint32_t key) {
      if ((key >> 8) == hi24) atomicAdd(&sh.hist[key & 0xffu], 1);
    });
  }
  __syncthreads();
  if (warp == 0) rt_pick(sh, 256, need);
  __syncthreads();
  const uint32_t T = (hi24 << 8) | (uint32_t)sh.bin;
  const int n_eq = need - sh.before;
  if (L <= kRtBitmapMax) {
    rt_place_bitmap(sh, rs, a, b, vec, T, n_eq, L, out, position);
    return;
  }
  // ---- placement: each warp's kept entries, counted, then written in order
  int gt = 0, eq = 0;
  rt_walk(rs, a, b, vec, [&](long long, uint32_t key) {
    gt += key > T;
    eq += key == T;
  });
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    gt += __shfl_xor_sync(0xffffffffu, gt, o);
    eq += __shfl_xor_sync(0xffffffffu, eq, o);
  }
  if (lane == 0) {
    sh.warp_gt[warp] = gt;
    sh.warp_eq[warp] = eq;
  }
  __syncthreads();
  int base = 0, eq_before = 0;
  for (int w = 0; w < warp; ++w) {
    eq_before += sh.warp_eq[w];
    base += sh.warp_gt[w] + max(0, min(sh.warp_eq[w], n_eq - (eq_before - sh.warp_eq[w])));
  }
  // in order: 32 (or 128) entries per step, ballots place them
  int eq_seen = 0;
  const unsigned lt = lanemask_lt();
  auto emit = [&](long long i, uint32_t key, bool valid) {
    const bool is_gt = valid && key > T, is_eq = valid && key == T;
    const unsigned em = __ballot_sync(0xffffffffu, is_eq);
    const bool keep = is_gt || (is_eq && eq_before + eq_seen + __popc(em & lt) < n_eq);
    const unsigned km = __ballot_sync(0xffffffffu, keep);
    if (keep) out[base + __popc(km & lt)] = position(i);
    base += __popc(km);
    eq_seen += __popc(em);
  };
  if (vec) {
    for (long long i0 = a; i0 < b; i0 += 128) {
      // lane l holds entries i0 + 4l .. +3; emit them in order: step u covers entries
      // i0 + 4l + u for every lane, which is not position order across lanes, so the four
      // are emitted one at a time after a transpose through shuffles
      float v4[4];
      const long long i = i0 + 4 * lane;
#pragma unroll
      for (int u = 0; u < 4; ++u) v4[u] = i + u < b ? rs[i + u] : 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        // entry i0 + 32u + lane sits in lane (32u + lane) / 4, slot (32u + lane) % 4
        const int src = (32 * u + lane) >> 2, slot = (32 * u + lane) & 3;
        const float x0 = __shfl_sync(0xffffffffu, v4[0], src), x1 = __shfl_sync(0xffffffffu, v4[1], src);
        const float x2 = __shfl_sync(0xffffffffu, v4[2], src), x3 = __shfl_sync(0xffffffffu, v4[3], src);
        const float x = slot == 0 ? x0 : slot == 1 ? x1 : slot == 2 ? x2 : x3;
        const long long e = i0 + 32 * u + lane;
        emit(e, score_key(x), e < b);
      }
    }
  } else {
    for (long long i0 = a; i0 < b; i0 += 32) {
      const long long i = i0 + lane;
      emit(i, i < b ? score_key(rs[i]) : 0u, i < b);
    }
  }
}

// A record range's candidate list: the selected columns idx[row] (ascending, -1 padded) to
// their scores and record positions (offset + column); one warp per row.
__global__ void shard_list_kernel(int n_rows, int K, const int32_t* idx, const float* scores, long long stride,
                                  long long offset, float* out_scores, int32_t* out_pos, int32_t* out_cnt) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= n_rows) return;
  int n = 0;
#pragma unroll 1
  for (int i = lane; i < K; i += 32) {
    const int32_t j = idx[(size_t)row * K + i];
    const bool ok = j >= 0;
    out_scores[(size_t)row * K + i] = ok ? scores[(size_t)row * stride + j] : -INFINITY;
    out_pos[(size_t)row * K + i] = ok ? (int32_t)(offset + j) : -1;
    n += ok;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
  if (lane == 0) out_cnt[row] = n;
}

// Gathered candidate lists, list-major [n_lists, n_rows, k_in] (and counts [n_lists, n_rows]),
// to the list merge's row-major order: keys (order-preserving images of the scores), positions
// and counts.
__global__ void lists_to_rows_kernel(int n_rows, int n_lists, int k_in, const float* scores, const int32_t* pos,
                                     const int32_t* cnt, uint32_t* keys, int32_t* pos_out, int32_t* cnt_out) {
  const long long n = (long long)n_rows * n_lists * k_in;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int k = (int)(i % k_in);
    const long long lr = i / k_in;
    const int r = (int)(lr % n_rows), l = (int)(lr / n_rows);  // source: list l, row r
    const size_t o = ((size_t)r * n_lists + l) * k_in + k;
    keys[o] = score_key(scores[i]);
    pos_out[o] = pos[i];
    if (k == 0) cnt_out[(size_t)r * n_lists + l] = cnt[lr];
  }
}

}  // namespace

cudaError_t launch_row_topk(const FeedParams& p, cudaStream_t stream) {
  if (p.n_rows == 0) return cudaSuccess;
  row_topk_kernel<<<p.n_rows, kRtThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_shard_list(int n_rows, int K, const int32_t* idx, const float* scores, long long stride,
                              long long offset, float* out_scores, int32_t* out_pos, int32_t* out_cnt,
                              cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  shard_list_kernel<<<(n_rows + 7) / 8, 256, 0, stream>>>(n_rows, K, idx, scores, stride, offset, out_scores, out_pos,
                                                          out_cnt);
  return cudaGetLastError();
}

cudaError_t launch_lists_to_rows(int n_rows, int n_lists, int k_in, const float* scores, const int32_t* pos,
                                 const int32_t* cnt, uint32_t* keys, int32_t* pos_out, int32_t* cnt_out,
                                 cudaStream_t stream) {
  const long long n = (long long)n_rows * n_lists * k_in;
  if (n == 0) return cudaSuccess;
  const long long blocks = std::min<long long>((n + 255) / 256, 4096);
  lists_to_rows_kernel<<<(int)blocks, 256, 0, stream>>>(n_rows, n_lists, k_in, scores, pos, cnt, keys, pos_out, cnt_out);
  return cudaGetLastError();
}

cudaError_t launch_lists_merge(const FeedParams& p, cudaStream_t stream) {
  if (p.n_rows == 0) return cudaSuccess;
  const int n_cta = std::min(kMergeMaxCta, std::max(2, p.in_seg));
  const int per = (p.in_seg + n_cta - 1) / n_cta;
  const size_t smem = merge_smem_bytes(per, p.in_K, p.K);
  if (p.in_seg > kMergeMaxLists || p.K > CSA2_MAX_TOPK || per * p.in_K >= 65536 || smem > 160u * 1024u)
    return launch_topk_feed(p, true, 1, stream);  // beyond the staged segment table or shared memory
  cudaError_t e = cudaFuncSetAttribute(lists_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_cta, p.n_rows);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)n_cta;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, lists_merge_kernel, p, per);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

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


}  // namespace csa2
