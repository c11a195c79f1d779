// Exact top-K of materialised rows and the merge of per-segment lists (the streaming
// engine of select.cuh fed from global memory), and the expansion of kept blocks into the
// hierarchical candidate pool ("DeepSeek-V4.1-Flash explained", section 3: a block is
// scored by its best position and every position of a kept block enters the pool).
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

// Merge of per-segment lists (source B) into a row's final top-K, one block per row.  The
// row's list keys are staged once in shared memory (keys below the largest per-segment K-th key
// zeroed: that segment alone holds K entries at or above it), then histogram passes run there.
// The candidates are a row's best keys and share their leading bits, so the levels are taken
// on the bits below the highest bit in which the smallest and largest candidate differ (a
// 12-bit window, then the next 12, then the rest): the level-1 bins spread the candidates
// instead of piling them onto a few counters.  One pass then counts per warp what it keeps
// and one writes the kept entries' list slots in order; the row's indices are those slots'
// positions.  Warp w owns a contiguous range of segments, so warp order followed by slot order
// is position order.
constexpr int kMergeWarps = 12;
constexpr int kMergeThreads = kMergeWarps * 32;
constexpr size_t kMergeSmemMax = 200u * 1024u;

__global__ void __launch_bounds__(kMergeThreads, 1) lists_merge_kernel(const FeedParams p) {
  extern __shared__ __align__(16) uint32_t kv[];  // [in_seg * in_K]
  __shared__ ArrSelShared sh;
  __shared__ int32_t sel_f[CSA2_MAX_TOPK];
  __shared__ uint32_t kext[2];  // smallest and largest candidate key
  ArrSel<kMergeWarps> s;
  s.sh = &sh;
  s.tid = threadIdx.x;
  const int row = blockIdx.x, S = p.in_seg, Kin = p.in_K, K = p.K;
  const int w = s.warp(), ln = s.lane();
  int* cnt = reinterpret_cast<int*>(sh.aux);  // [S <= 64]
  uint32_t* thr_s = sh.aux + 64;
  for (int i = s.tid; i < S; i += kMergeThreads) {
    cnt[i] = min(__ldcg(p.in_cnt + (size_t)row * S + i), Kin);
    thr_s[i] = p.in_thr ? __ldcg(p.in_thr + (size_t)row * S + i) : 0u;
  }
  if (s.tid == 0) kext[0] = 0xffffffffu, kext[1] = 0u;
  s.zero_hist(kHistBins);
  s.sync();
  uint32_t thr0 = 0u;
  for (int i = 0; i < S; ++i) thr0 = max(thr0, thr_s[i]);
  const int n = S * Kin;
  const uint32_t* gk = p.in_keys + (size_t)row * n;
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  auto filt = [&](uint32_t key, int sg, int j) -> uint32_t {
    key = (j < cnt[sg] && key >= thr0) ? key : 0u;
    if (key) kmin = min(kmin, key), kmax = max(kmax, key);
    return key;
  };
  if ((Kin & 3) == 0) {
    const uint4* g4 = reinterpret_cast<const uint4*>(gk);
    uint4* s4 = reinterpret_cast<uint4*>(kv);
#pragma unroll 4
    for (int i = s.tid; i < n / 4; i += kMergeThreads) {
      uint4 v = __ldcg(g4 + i);
      const int sg = (4 * i) / Kin, j = 4 * i - sg * Kin;
      v.x = filt(v.x, sg, j), v.y = filt(v.y, sg, j + 1), v.z = filt(v.z, sg, j + 2), v.w = filt(v.w, sg, j + 3);
      s4[i] = v;
    }
  } else {
#pragma unroll 4
    for (int i = s.tid; i < n; i += kMergeThreads) kv[i] = filt(__ldcg(gk + i), i / Kin, i % Kin);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if (ln == 0 && kmax != 0u) atomicMin(&kext[0], kmin), atomicMax(&kext[1], kmax);
  s.sync();
  kmin = kext[0], kmax = kext[1];
  // bits above d are common to every candidate
  const int d = kmax > kmin ? 31 - __clz(kmin ^ kmax) : 0;
  const int s1 = max(d - 11, 0), s2 = max(s1 - 12, 0);
  const uint32_t m1 = (2u << (d - s1)) - 1u;
  for (int i = s.tid; i < n; i += kMergeThreads) {
    const uint32_t key = kv[i];
    if (key) atomicAdd(&sh.hist[(key >> s1) & m1], 1);
  }
  s.sync();
  s.template pick<kHistBins>(K);
  uint32_t thr = 0u;
  int n_eq = 0;
  if (sh.total > K) {
    // T: the threshold's bits above the current shift
    uint32_t T = ((kmax >> s1) & ~m1) | (uint32_t)sh.bin;
    int need = K - sh.before;
    if (s1 > 0) {
      const uint32_t m2 = (1u << (s1 - s2)) - 1u;
      s.sync();
      s.zero_hist(kHistBins);
      s.sync();
      for (int i = s.tid; i < n; i += kMergeThreads) {
        const uint32_t key = kv[i];
        if (key && (key >> s1) == T) atomicAdd(&sh.hist[(key >> s2) & m2], 1);
      }
      s.sync();
      s.template pick<kHistBins>(need);
      T = (T << (s1 - s2)) | (uint32_t)sh.bin;
      need -= sh.before;
      if (s2 > 0) {
        const uint32_t m3 = (1u << s2) - 1u;  // s2 <= 8
        s.sync();
        s.zero_hist(256);
        s.sync();
        for (int i = s.tid; i < n; i += kMergeThreads) {
          const uint32_t key = kv[i];
          if (key && (key >> s2) == T) atomicAdd(&sh.hist[key & m3], 1);
        }
        s.sync();
        s.template pick<256>(need);
        T = (T << s2) | (uint32_t)sh.bin;
        need -= sh.before;
      }
    }
    thr = T;
    n_eq = need;
  }
  // warp w: slots [f0, f1) of whole segments, in order
  const int f0 = (int)(((long long)S * w) / kMergeWarps) * Kin, f1 = (int)(((long long)S * (w + 1)) / kMergeWarps) * Kin;
  int gt = 0, eq = 0;
  for (int f = f0 + ln; f < f1; f += 32) {
    const uint32_t key = kv[f];
    gt += key != 0u && key > thr;
    eq += key != 0u && key == thr;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    gt += __shfl_xor_sync(0xffffffffu, gt, o);
    eq += __shfl_xor_sync(0xffffffffu, eq, o);
  }
  // gt <= K in every warp and in sum; equal keys beyond K per warp never change what is taken,
  // so clamping keeps both halves of the packed scan below 2^16
  eq = min(eq, K);
  int tot_packed;
  const int before = s.scan(ln == 0 ? (gt << 16) | eq : 0, &tot_packed);
  const int pb = __shfl_sync(0xffffffffu, before, 0);
  const int eq_b = pb & 0xffff;
  const int take = max(0, min(eq, n_eq - eq_b));
  int base = (pb >> 16) + min(eq_b, n_eq);
  const int kept = min(K, (tot_packed >> 16) + min(tot_packed & 0xffff, n_eq));
  int eq_seen = 0;
  const unsigned lt = lanemask_lt();
  for (int f0r = f0; f0r < f1; f0r += 32) {  // warp-uniform trip count
    const int f = f0r + ln;
    const uint32_t key = f < f1 ? kv[f] : 0u;
    const bool is_eq = key != 0u && key == thr;
    const unsigned em = __ballot_sync(0xffffffffu, is_eq);
    const bool keep = key != 0u && (key > thr || (is_eq && eq_seen + __popc(em & lt) < take));
    const unsigned km = __ballot_sync(0xffffffffu, keep);
    const int r = base + __popc(km & lt);
    if (keep && r < K) sel_f[r] = f;
    base += __popc(km);
    eq_seen += __popc(em);
  }
  s.sync();
  const int32_t* pos = p.in_pos + (size_t)row * n;
  int32_t* out = p.idx + (size_t)row * K;
  for (int r = s.tid; r < K; r += kMergeThreads) out[r] = r < kept ? __ldcg(pos + sel_f[r]) : -1;
}

}  // namespace

cudaError_t launch_lists_merge(const FeedParams& p, cudaStream_t stream) {
  if (p.n_rows == 0) return cudaSuccess;
  const size_t smem = (size_t)p.in_seg * p.in_K * sizeof(uint32_t);
  if (p.in_seg > 64 || p.K > CSA2_MAX_TOPK || smem > kMergeSmemMax)
    return launch_topk_feed(p, true, 1, stream);  // beyond the staged segment table or shared memory
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(lists_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMergeSmemMax);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  lists_merge_kernel<<<p.n_rows, kMergeThreads, smem, stream>>>(p);
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

cudaError_t launch_pool_expand(const int32_t* kept, const int32_t* n_visible, int n_rows, int n_keep,
                               int block_size, int32_t* pool, int32_t* n_pool, cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  pool_expand_kernel<<<n_rows, 256, 0, stream>>>(kept, n_visible, n_keep, block_size, pool, n_pool);
  return cudaGetLastError();
}

}  // namespace csa2
