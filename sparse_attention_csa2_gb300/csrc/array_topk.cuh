// Exact top-K of an array of keys held in shared memory, in entry order, by the NW warps of a
// thread block.
//
// Rule (course lesson "06 / Indexer and attention", select_values and its note on ties): the
// K entries best by (key descending, entry index ascending) are kept; keys are the
// order-preserving images of the scores (score_key), 0 marks an entry that is not a
// candidate.
//
// The K-th key is found with three histogram levels over the key bits 31..20, 19..8 and 7..0.
// Each warp owns a contiguous range of the array.  After the first level a single pass over
// the array copies, per warp and in entry order, every entry whose key is at or above the
// threshold's level-1 bin (key and index) to a list in scratch memory.  The two finer levels,
// the counts and the output all walk those lists only, which hold about K entries plus the
// population of one bin, so the array is read once after its histogram.  The first level's
// histogram may be filled by the caller while the keys are produced.
//
// The selection runs once per thread block, so its code is never warm in the instruction
// cache: the functions are kept out of line (every caller in a kernel shares one copy) and
// their loops rolled.
#pragma once

#include "common.cuh"

namespace csa2 {

constexpr int kHistBins = 4096;

struct alignas(16) ArrSelShared {
  int hist[kHistBins];
  int tmp[32];
  int w_list[32];     // per warp: entries in its list
  uint32_t aux[128];  // free for the caller between selections
  int bin;            // chosen bin of the current level
  int before;         // candidates above it
  int total;
  uint32_t thr;       // the K-th key (0 when at most K candidates)
  int n_eq;           // entries equal to thr that are kept, lowest indices first
};

// hist[bin] += 1 when `valid`.  A plain shared atomic: on sm_103a aggregating equal bins over
// the warp first (match.any) costs far more than the atomics' own serialisation, even when
// every lane hits the same bin.
__device__ __forceinline__ void hist_add(int* hist, uint32_t bin, bool valid) {
  if (valid) atomicAdd(&hist[bin], 1);
}

template <int NW>
struct ArrSel {
  static constexpr int NT = NW * 32;
  ArrSelShared* sh;
  int tid;
  uint32_t* scratch = nullptr;  // per-warp lists, list_words(n) words, 16-byte aligned

  __device__ __forceinline__ void sync() const { __syncthreads(); }
  __device__ __forceinline__ int lane() const { return tid & 31; }
  __device__ __forceinline__ int warp() const { return tid >> 5; }

  // Entries of the array owned by each warp (a multiple of 128, so every warp's range starts
  // on a 16-byte boundary and is read in whole 128-entry steps).
  __host__ __device__ static constexpr int range(int n) { return ((n + NW - 1) / NW + 127) & ~127; }
  // Scratch words the lists of an n-entry array take.
  __host__ __device__ static constexpr int list_words(int n) { return 2 * NW * range(n); }

  // Exclusive prefix sum over the group in thread order; *total gets the sum.
  __device__ __forceinline__ int scan(int v, int* total) const {
    const int ln = lane(), w = warp();
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (ln >= o) x += y;
    }
    if (ln == 31) sh->tmp[w] = x;
    sync();
    int before = 0, tot = 0;
#pragma unroll
    for (int v2 = 0; v2 < NW; ++v2) {
      const int c = sh->tmp[v2];
      before += v2 < w ? c : 0;
      tot += c;
    }
    *total = tot;
    sync();
    return before + x - v;
  }

  __device__ __forceinline__ void zero_hist(int nbins) const {
    for (int i = tid; i < nbins; i += NT) sh->hist[i] = 0;
  }

  // Finds the bin, searched from the top, at which the count from above first reaches `need`:
  // sh->bin and sh->before (the count above it); sh->total gets the sum of all bins.  Each
  // thread takes an odd number of consecutive bins (no bank conflicts), holds them in
  // registers, and the thread whose share holds the crossing finds it there.  `h`: the
  // histogram (sh->hist when null).
  template <int NBINS>
  __device__ __noinline__ void pick(int need, const int* h = nullptr) const {
    constexpr int PER = ((NBINS + NT - 1) / NT) | 1;
    const int* hist = h ? h : sh->hist;
    const int r0 = tid * PER;  // rank from the top of this thread's first bin
    int c[PER];
    int local = 0;
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      c[q] = r0 + q < NBINS ? hist[NBINS - 1 - (r0 + q)] : 0;
      local += c[q];
    }
    int tot;
    const int before = scan(local, &tot);
    if (before < need && before + local >= need) {
      int acc = before;
      bool found = false;
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        if (!found && acc + c[q] >= need) {
          found = true;
          sh->bin = NBINS - 1 - (r0 + q);
          sh->before = acc;
        }
        acc += c[q];
      }
    }
    if (tid == 0) sh->total = tot;
    sync();
  }
};

// Finds the K-th key of keys[0..n) (0 = not a candidate) and lists the candidates at or
// above its level-1 bin.  `keys` is 16-byte aligned and readable up to n rounded up to a
// multiple of 4.  `hist_ready`: the caller has filled sh->hist with the level-1 histogram
// (key >> 20) of the candidates.  Afterwards sh->thr and sh->n_eq describe the selection:
// keys > thr, and the first n_eq keys == thr in entry order (thr = 0, n_eq = 0 when at most k
// candidates exist: all are kept).
// The histogram levels' bin choice, for a block on its own: the block's histogram.
template <int NW>
struct LocalPick {
  template <int NBINS>
  __device__ __forceinline__ void run(const ArrSel<NW>& s, int need) const {
    s.template pick<NBINS>(need);
  }
  // Levels 2 (bits 19..8) and 3 (bits 7..0) over the warp lists' keys in bin b1; sets
  // sh->thr and sh->n_eq.
  __device__ __forceinline__ void refine(const ArrSel<NW>& s, const uint32_t* lk, int n_list, uint32_t b1,
                                         int need, uint32_t* local_keys) const {
    (void)local_keys;
    ArrSelShared& sh = *s.sh;
    const int ln = s.lane();
    s.zero_hist(kHistBins);
    s.sync();
#pragma unroll 1
    for (int j = ln; j < n_list; j += 32)
      if ((lk[j] >> 20) == b1) atomicAdd(&sh.hist[(lk[j] >> 8) & 0xfffu], 1);
    s.sync();
    s.template pick<kHistBins>(need);
    const uint32_t hi24 = (b1 << 12) | (uint32_t)sh.bin;
    need -= sh.before;
    s.sync();
    s.zero_hist(256);
    s.sync();
#pragma unroll 1
    for (int j = ln; j < n_list; j += 32)
      if ((lk[j] >> 8) == hi24) atomicAdd(&sh.hist[lk[j] & 0xffu], 1);
    s.sync();
    s.template pick<256>(need);
    if (s.tid == 0) {
      sh.thr = (hi24 << 8) | (uint32_t)sh.bin;
      sh.n_eq = need - sh.before;
    }
    s.sync();
  }
};

// The bin choice for the blocks of a thread-block cluster that select over the union of their
// arrays (the segments of one row): block 0 adds the others' histograms into its own (through
// distributed shared memory), picks, and writes bin / before / total into every block.  All
// blocks of the cluster call it at the same points.
template <int NW>
struct ClusterPick {
  uint32_t rank, n_cta;
  int local_cap;  // capacity of block 0's key array (words) for the keys of bin b1
  // Level 1: every block adds one slice of the bins over the cluster into block 0's
  // histogram, block 0 picks and writes bin / before / total into every block.
  template <int NBINS>
  __device__ __forceinline__ void run(const ArrSel<NW>& s, int need) const {
    constexpr int NT = NW * 32;
    ArrSelShared& sh = *s.sh;
    cluster_sync();  // every block's histogram is final
    const int n_v4 = NBINS / 4, per = (n_v4 + (int)n_cta - 1) / (int)n_cta;
    const int lo = (int)rank * per, hi = min(n_v4, lo + per);
#pragma unroll 1
    for (int i = lo + s.tid; i < hi; i += NT) {
      uint4 acc = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 4
      for (uint32_t c = 0; c < n_cta; ++c) {
        const uint4 v = cluster_ld_v4(cluster_map(&sh.hist[4 * i], c));
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      cluster_st_v4(cluster_map(&sh.hist[4 * i], 0), acc);
    }
    cluster_sync();  // block 0 holds the cluster's histogram
    if (rank == 0) {
      s.template pick<NBINS>(need);
      if (s.tid > 0 && (uint32_t)s.tid < n_cta) {
        cluster_st_s32(cluster_map(&sh.bin, s.tid), sh.bin);
        cluster_st_s32(cluster_map(&sh.before, s.tid), sh.before);
        cluster_st_s32(cluster_map(&sh.total, s.tid), sh.total);
      }
    }
    cluster_sync();  // the choice is visible in every block; the histograms may be reused
  }
  // Levels 2 and 3 by block 0 alone over every block's listed keys in bin b1 (few): warp w of
  // block 0 gathers list w of every block through distributed shared memory (lane c first
  // reads block c's list length and layout, then the lanes take the concatenated lists'
  // entries in strides), keeps the keys in bin b1 with their block in its own key array (free
  // once its lists exist) and counts level 2; level 3 reads that local copy.  Block 0 then
  // knows, per block, how many of its entries lie above the threshold and how many equal it,
  // and writes into every block its threshold, its number of tied entries to keep (n_eq), its
  // row offset (aux[2]) and the row's number of selected entries (aux[4]).  Each block has
  // published its warps' list lengths (w_list) and its range per warp (aux[5]).
  __device__ __forceinline__ void refine(const ArrSel<NW>& s, const uint32_t* lk, int n_list, uint32_t b1,
                                         int need, uint32_t* local_keys) const {
    (void)lk;
    (void)n_list;
    ArrSelShared& sh = *s.sh;
    const int w = s.warp(), ln = s.lane();
    uint32_t* cnt_all = sh.aux + 16;  // per block: listed entries
    uint32_t* cnt_gt = sh.aux + 32;   // ... above the threshold (bins above b1 included later)
    uint32_t* cnt_b1 = sh.aux + 48;   // ... in bin b1
    uint32_t* cnt_eq = sh.aux + 64;   // ... equal to the threshold
    const int cap = local_cap / 2;    // local copy: keys, then their blocks
    uint32_t* local_src = local_keys + cap;
    cluster_sync();  // every block's lists are complete
    if (rank == 0) {
      int my_len = 0, my_per = 0;
      if ((uint32_t)ln < n_cta) {
        my_len = cluster_ld_s32(cluster_map(&sh.w_list[w], ln));
        my_per = cluster_ld_s32(cluster_map(&sh.aux[5], ln));
      }
      int incl = my_len;  // inclusive prefix of the lists' lengths over the blocks
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (ln >= o) incl += y;
      }
      const int total = __shfl_sync(0xffffffffu, incl, 31);
      s.zero_hist(kHistBins);
      if (s.tid < 64) sh.aux[16 + s.tid] = 0u;
      if (s.tid == 0) sh.aux[6] = 0u;  // keys kept in bin b1
      s.sync();
      if ((uint32_t)ln < n_cta) atomicAdd(&cnt_all[ln], (uint32_t)my_len);
      const unsigned lt = lanemask_lt();
      // entry f of warp w's concatenated lists: its block and its key
      auto entry = [&](int f, int& c) -> uint32_t {
        int start = 0;
        c = 0;
#pragma unroll 1
        for (int q = 0; q < (int)n_cta; ++q) {
          const int end = __shfl_sync(0xffffffffu, incl, q);
          if (f >= end) {
            c = q + 1;
            start = end;
          }
        }
        const int per_c = __shfl_sync(0xffffffffu, my_per, min(c, (int)n_cta - 1));
        return f < total ? (uint32_t)cluster_ld_s32(
                               cluster_map(s.scratch + (size_t)w * 2 * per_c + (f - start), (uint32_t)min(c, (int)n_cta - 1)))
                         : 0u;
      };
#pragma unroll 1
      for (int f0 = 0; f0 < total; f0 += 32) {
        const int f = f0 + ln;
        int c;
        const uint32_t key = entry(f, c);
        const bool in = f < total && (key >> 20) == b1;
        const unsigned m = __ballot_sync(0xffffffffu, in);
        int base = 0;
        if (ln == 0 && m) base = (int)atomicAdd(&sh.aux[6], (uint32_t)__popc(m));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (in) {
          const int slot = base + __popc(m & lt);
          if (slot < cap) {
            local_keys[slot] = key;
            local_src[slot] = (uint32_t)c;
          }
          atomicAdd(&sh.hist[(key >> 8) & 0xfffu], 1);
          atomicAdd(&cnt_b1[c], 1u);
        }
      }
      s.sync();
      s.template pick<kHistBins>(need);
      const uint32_t hi24 = (b1 << 12) | (uint32_t)sh.bin;
      const int need3 = need - sh.before;
      const int n_b1 = (int)sh.aux[6];
      s.sync();
      s.zero_hist(256);
      s.sync();
      const bool local = n_b1 <= cap;
      if (local) {
#pragma unroll 1
        for (int j = s.tid; j < n_b1; j += NW * 32)
          if ((local_keys[j] >> 8) == hi24) atomicAdd(&sh.hist[local_keys[j] & 0xffu], 1);
      } else {  // more keys in bin b1 than the local copy holds: read the blocks' lists again
#pragma unroll 1
        for (int f0 = 0; f0 < total; f0 += 32) {
          int c;
          const uint32_t key = entry(f0 + ln, c);
          if (f0 + ln < total && (key >> 8) == hi24) atomicAdd(&sh.hist[key & 0xffu], 1);
        }
      }
      s.sync();
      s.template pick<256>(need3);
      const uint32_t thr = (hi24 << 8) | (uint32_t)sh.bin;
      const int n_eq_row = need3 - sh.before;
      // per block: its keys of bin b1 above the threshold and equal to it
      if (local) {
#pragma unroll 1
        for (int j = s.tid; j < n_b1; j += NW * 32) {
          if (local_keys[j] > thr) atomicAdd(&cnt_gt[local_src[j]], 1u);
          if (local_keys[j] == thr) atomicAdd(&cnt_eq[local_src[j]], 1u);
        }
      } else {
#pragma unroll 1
        for (int f0 = 0; f0 < total; f0 += 32) {
          int c;
          const uint32_t key = entry(f0 + ln, c);
          if (f0 + ln < total && (key >> 20) == b1) {
            if (key > thr) atomicAdd(&cnt_gt[c], 1u);
            if (key == thr) atomicAdd(&cnt_eq[c], 1u);
          }
        }
      }
      s.sync();
      if (w == 0) {
        // offsets in block order: every listed entry above bin b1 is kept, then those of bin
        // b1 above the threshold, then the first n_eq_row ties in block order
        int g = 0, e = 0;
        if ((uint32_t)ln < n_cta) {
          g = (int)(cnt_all[ln] - cnt_b1[ln] + cnt_gt[ln]);
          e = (int)cnt_eq[ln];
        }
        int gi = g, ei = e;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int yg = __shfl_up_sync(0xffffffffu, gi, o), ye = __shfl_up_sync(0xffffffffu, ei, o);
          if (ln >= o) {
            gi += yg;
            ei += ye;
          }
        }
        const int gb = gi - g, eb = ei - e;
        const int G = __shfl_sync(0xffffffffu, gi, 31), E = __shfl_sync(0xffffffffu, ei, 31);
        if ((uint32_t)ln < n_cta) {
          cluster_st_s32(cluster_map(&sh.thr, ln), (int)thr);
          cluster_st_s32(cluster_map(&sh.n_eq, ln), max(0, min(e, n_eq_row - eb)));
          cluster_st_s32(cluster_map(&sh.aux[2], ln), gb + min(eb, n_eq_row));
          cluster_st_s32(cluster_map(&sh.aux[4], ln), G + min(E, n_eq_row));
        }
      }
    }
    cluster_sync();  // thresholds and offsets are visible in every block
  }
};

template <int NW, class Pick>
__device__ __noinline__ void arr_threshold_impl(const ArrSel<NW>& s, const uint32_t* keys, int n, int k,
                                                bool hist_ready, Pick picker) {
  constexpr int NT = NW * 32;
  ArrSelShared& sh = *s.sh;
  const int w = s.warp(), ln = s.lane();
  if (!hist_ready) {
    s.zero_hist(kHistBins);
    s.sync();
#pragma unroll 1
    for (int i = s.tid; i < n; i += NT)
      if (keys[i] != 0u) atomicAdd(&sh.hist[keys[i] >> 20], 1);
    s.sync();
  }
  picker.template run<kHistBins>(s, k);
  const bool all = sh.total <= k;  // at most k candidates: keep them all
  const uint32_t b1 = all ? 0u : (uint32_t)sh.bin;
  int need = k - sh.before;
  const int per = ArrSel<NW>::range(n);
  s.sync();  // every thread has read bin / before / total
  uint32_t* lk = s.scratch + (size_t)w * 2 * per;  // keys of the warp's list
  uint32_t* li = lk + per;                         // their entry indices
  // Lane l of the warp owns entries [lo + l*q, lo + (l+1)*q) of the warp's range (q = per/32,
  // a multiple of 4).  A first walk counts the lane's entries at or above bin b1, one warp
  // scan places each lane's share in the list, and a second walk writes them: the list is in
  // entry order, and the walks are plain vector loads with no warp votes.
  int n_list;
  {
    const int lo = min(n, w * per), hi = min(n, lo + per);
    const int q = per / 32;
    const int a0 = min(hi, lo + ln * q), a1 = min(hi, a0 + q);
    auto listed = [&](uint32_t key) { return key != 0u && (key >> 20) >= b1; };
    int c = 0;
#pragma unroll 1
    for (int i = a0; i < a1; i += 4) {
      const uint4 v = *reinterpret_cast<const uint4*>(keys + i);
      c += listed(v.x) + (i + 1 < a1 && listed(v.y)) + (i + 2 < a1 && listed(v.z)) + (i + 3 < a1 && listed(v.w));
    }
    int inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, o);
      if (ln >= o) inc += y;
    }
    n_list = __shfl_sync(0xffffffffu, inc, 31);
    int at = inc - c;
#pragma unroll 1
    for (int i = a0; c > 0 && i < a1; i += 4) {
      const uint4 v = *reinterpret_cast<const uint4*>(keys + i);
      const uint32_t kv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i + u < a1 && listed(kv[u])) {
          lk[at] = kv[u];
          li[at] = (uint32_t)(i + u);
          ++at;
          --c;
        }
    }
    if (ln == 0) sh.w_list[w] = n_list;
  }
  if (s.tid == 0) sh.aux[5] = (uint32_t)per;  // the lists' layout, for a cluster's block 0
  if (all) {
    if (s.tid == 0) {
      sh.thr = 0u;
      sh.n_eq = 0;
    }
    s.sync();
    return;
  }
  s.sync();
  picker.refine(s, lk, n_list, b1, need, const_cast<uint32_t*>(keys));
}

template <int NW>
__device__ __forceinline__ void arr_threshold(const ArrSel<NW>& s, const uint32_t* keys, int n, int k,
                                              bool hist_ready) {
  arr_threshold_impl(s, keys, n, k, hist_ready, LocalPick<NW>{});
}

// Writes the entry indices of the selected entries, in entry order, to sel[0 .. kept) and
// returns kept.  Follows arr_threshold on the same n and group with the lists untouched in
// between.  n < 65536.
template <int NW>
__device__ __noinline__ int arr_compact(const ArrSel<NW>& s, int n, int32_t* sel) {
  ArrSelShared& sh = *s.sh;
  const uint32_t thr = sh.thr;
  const int n_eq = sh.n_eq;
  const int w = s.warp(), ln = s.lane();
  const unsigned lt = lanemask_lt();
  const int per = ArrSel<NW>::range(n);
  const uint32_t* lk = s.scratch + (size_t)w * 2 * per;
  const uint32_t* li = lk + per;
  const int len = sh.w_list[w];
  int gt = 0, eq = 0;
#pragma unroll 1
  for (int j = ln; j < len; j += 32) {
    gt += lk[j] > thr;
    eq += lk[j] == thr;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    gt += __shfl_xor_sync(0xffffffffu, gt, o);
    eq += __shfl_xor_sync(0xffffffffu, eq, o);
  }
  // One scan of the warps' counts packed in one int (above thr in the high half, equal in the
  // low half): the entries equal to thr are taken in warp order, so a warp's output starts
  // after the entries above thr of the warps before it and the taken equal ones among theirs.
  int tot_packed;
  const int before = s.scan(ln == 0 ? (gt << 16) | eq : 0, &tot_packed);  // lane 0 carries the counts
  const int pb = __shfl_sync(0xffffffffu, before, 0);
  const int eq_b = pb & 0xffff;
  const int take = max(0, min(eq, n_eq - eq_b));
  int base = (pb >> 16) + min(eq_b, n_eq);
  const int tot = (tot_packed >> 16) + min(tot_packed & 0xffff, n_eq);
  int eq_seen = 0;
#pragma unroll 1
  for (int j0 = 0; j0 < len; j0 += 32) {
    const int j = j0 + ln;
    const uint32_t key = j < len ? lk[j] : 0u;
    const bool is_eq = key != 0u && key == thr;
    const unsigned em = __ballot_sync(0xffffffffu, is_eq);
    const bool keep = key != 0u && (key > thr || (is_eq && eq_seen + __popc(em & lt) < take));
    const unsigned km = __ballot_sync(0xffffffffu, keep);
    if (keep) sel[base + __popc(km & lt)] = (int32_t)li[j];
    base += __popc(km);
    eq_seen += __popc(em);
  }
  s.sync();
  return tot;
}

// Cluster mode (the blocks of a cluster select over the union of their arrays, in block order):
// after arr_threshold_impl with ClusterPick, each block publishes how many of its listed
// entries lie above the threshold and how many equal it; the entries equal to the threshold
// are taken in block order, then entry order.  Writes this block's selected entries (entry
// indices, in order) to sel and returns their number; *base gets the row offset of the first,
// *total the row's number of selected entries.
template <int NW>
__device__ __noinline__ int arr_compact_cluster(const ArrSel<NW>& s, int n, int32_t* sel, uint32_t rank,
                                                uint32_t n_cta, int* base, int* total) {
  ArrSelShared& sh = *s.sh;
  const uint32_t thr = sh.thr;
  const int n_eq = sh.n_eq;
  const int w = s.warp(), ln = s.lane();
  const int per = ArrSel<NW>::range(n);
  const uint32_t* lk = s.scratch + (size_t)w * 2 * per;
  const int len = sh.w_list[w];
  int gt = 0, eq = 0;
#pragma unroll 1
  for (int j = ln; j < len; j += 32) {
    gt += lk[j] > thr;
    eq += lk[j] == thr;
  }
  int tot;
  const int packed_before = s.scan((gt << 16) | eq, &tot);  // per-thread packed counts
  (void)packed_before;
  if (s.tid == 0) {
    sh.aux[0] = (uint32_t)(tot >> 16);     // above the threshold in this block
    sh.aux[1] = (uint32_t)(tot & 0xffff);  // equal to it
  }
  cluster_sync();  // every block's counts are published
  if (w == 0) {
    int g = 0, e = 0;
    if ((uint32_t)ln < n_cta) {
      g = cluster_ld_s32(cluster_map(&sh.aux[0], ln));
      e = cluster_ld_s32(cluster_map(&sh.aux[1], ln));
    }
    int gb = (uint32_t)ln < rank ? g : 0, eb = (uint32_t)ln < rank ? e : 0, G = g, E = e;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      gb += __shfl_xor_sync(0xffffffffu, gb, o);
      eb += __shfl_xor_sync(0xffffffffu, eb, o);
      G += __shfl_xor_sync(0xffffffffu, G, o);
      E += __shfl_xor_sync(0xffffffffu, E, o);
    }
    const int e_mine = __shfl_sync(0xffffffffu, e, (int)rank);
    if (ln == 0) {
      sh.aux[2] = (uint32_t)(gb + min(eb, n_eq));
      sh.aux[3] = (uint32_t)max(0, min(e_mine, n_eq - eb));
      sh.aux[4] = (uint32_t)(G + min(E, n_eq));
    }
  }
  cluster_sync();  // every block has read the others' counts
  if (s.tid == 0) sh.n_eq = (int)sh.aux[3];
  s.sync();
  *base = (int)sh.aux[2];
  *total = (int)sh.aux[4];
  return arr_compact(s, n, sel);
}

}  // namespace csa2
