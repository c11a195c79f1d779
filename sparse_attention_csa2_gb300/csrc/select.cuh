// Exact streaming top-K of one row, run by a group of NW warps of a thread block.
//
// Selection rule (course lesson "06 / Indexer and attention", select_values, and its note on
// ties): keep the K entries that are best by (score descending, entry index ascending).
// Scores are compared through order-preserving uint32 keys (score_key), so -0.0 == +0.0
// and every comparison is exact.
//
// Every warp of the group owns a buffer of (key, entry index j) pairs, in any order.  A
// warp appends the entries of each 32-lane group whose key is at least `thr` with a ballot.
// `thr` is the K-th best key among the entries kept so far (0 until K entries have been
// seen): an entry with a smaller key ranks behind K others whatever its index, so it can
// be dropped in any feeding order; ties with thr are kept and decided by index at the next
// select.  When a buffer nears capacity the group runs `eng_select`: an
// MSB-first 8-bit radix select finds the K-th key thr and how many entries equal to it to
// keep; if that is fewer than all of them, a second radix select over the indices of the
// tied entries finds the last index to keep.  Each warp then compacts its buffer.
// Feeders append each warp's entries in ascending index order and compaction keeps order, so
// every buffer stays sorted by index; `eng_finish` merges them by binary search.
#pragma once

#include "common.cuh"

namespace csa2 {

constexpr int kRoundEntries = 128;  // most entries one warp appends between two checks
constexpr int kEngMaxWarps = 16;
constexpr int kEngMaxK = 1024;

struct EngShared {
  int hist[256];
  int tmp[32];
  int warp_cnt[kEngMaxWarps];
  uint32_t thr;
  int sel_digit;
  int sel_before;
  int sel_count;
  uint32_t all_and;  // AND / OR of every key: bits where they agree need no radix pass
  uint32_t all_or;
};

// Histogram increment; `bin` < 0 adds nothing.  A plain shared atomic: on sm_103a
// aggregating equal bins over the warp first (match.any) costs far more than the atomics' own
// serialisation, even when every lane hits the same bin.
__device__ __forceinline__ void warp_hist_add(int* hist, int bin) {
  if (bin >= 0) atomicAdd(&hist[bin], 1);
}

template <int NW>
struct Engine {
  static constexpr int NT = NW * 32;
  uint32_t* keys;     // [NW * cap]
  int32_t* js;        // [NW * cap] entry indices
  uint32_t* out_key;  // [K] emission scratch
  int32_t* out_j;     // [K]
  int cap;            // per-warp capacity, >= K + kRoundEntries
  EngShared* sh;
  int bar_id;         // 0: __syncthreads (the group is the whole block); else a named barrier
  int tid;            // 0 .. NT-1 within the group

  __device__ __forceinline__ void sync() const {
    if (bar_id == 0)
      __syncthreads();
    else
      asm volatile("bar.sync %0, %1;\n" ::"r"(bar_id), "n"(NT) : "memory");
  }
  __device__ __forceinline__ int lane() const { return tid & 31; }
  __device__ __forceinline__ int warp() const { return tid >> 5; }

  // Exclusive prefix sum over the group; *total gets the sum.
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
    if (w == 0) {
      int t = ln < NW ? sh->tmp[ln] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, t, o);
        if (ln >= o) t += y;
      }
      if (ln < NW) sh->tmp[ln] = t;
    }
    sync();
    const int before = w ? sh->tmp[w - 1] : 0;
    *total = sh->tmp[NW - 1];
    sync();
    return before + x - v;
  }
};

template <int NW>
__device__ __forceinline__ void eng_init(const Engine<NW>& e, uint32_t thr0 = 0u) {
  if (e.tid < NW) e.sh->warp_cnt[e.tid] = 0;
  if (e.tid == 0) e.sh->thr = thr0;
  e.sync();
}

// Appends, as one 32-lane group, the lanes' entries that are valid with key >= thr.
// `cnt` is this warp's fill (warp-uniform).  The caller guarantees room for 32 more.
template <int NW>
__device__ __forceinline__ void eng_append(const Engine<NW>& e, int& cnt, uint32_t thr, bool valid, uint32_t key,
                                           int32_t j) {
  const bool keep = valid && key >= thr && key != 0u;
  const unsigned m = __ballot_sync(0xffffffffu, keep);
  if (keep) {
    const int o = e.warp() * e.cap + cnt + __popc(m & lanemask_lt());
    e.keys[o] = key;
    e.js[o] = j;
  }
  cnt += __popc(m);
}

// One radix digit search over sh->hist: the digit at which the running count (from the top
// digit down when `desc`, else from digit 0 up) first reaches `need`.  Stores the digit, the
// count before it and its own count in sh.
template <int NW>
__device__ __forceinline__ void eng_pick_digit(const Engine<NW>& e, int need, bool desc) {
  constexpr int NT = NW * 32;
  constexpr int BPT = NT >= 256 ? 1 : 256 / NT;  // bins per thread
  const int t = e.tid;
  int h[BPT];
  int local = 0;
#pragma unroll
  for (int k = 0; k < BPT; ++k) {
    const int r = t * BPT + k;  // rank of the bin in search order
    h[k] = r < 256 ? e.sh->hist[desc ? 255 - r : r] : 0;
    local += h[k];
  }
  int tot;
  int before = e.scan(local, &tot);
#pragma unroll
  for (int k = 0; k < BPT; ++k) {
    const int r = t * BPT + k;
    if (r < 256 && before < need && before + h[k] >= need) {
      e.sh->sel_digit = desc ? 255 - r : r;
      e.sh->sel_before = before;
      e.sh->sel_count = h[k];
    }
    before += h[k];
  }
  e.sync();
}

// Keeps the top-k of the group's buffers.  Updates warp counts and sh->thr.  All threads of
// the group must call it.
template <int NW>
__device__ __noinline__ void eng_select(const Engine<NW> e, int k) {
  constexpr int NT = NW * 32;
  EngShared& s = *e.sh;
  const int t = e.tid, ln = e.lane(), w = e.warp();
  const int mycnt = s.warp_cnt[w];
  int total = 0;
#pragma unroll
  for (int i = 0; i < NW; ++i) total += s.warp_cnt[i];
  if (total <= k) {
    e.sync();
    return;
  }
  uint32_t* kb = e.keys + w * e.cap;
  int32_t* jb = e.js + w * e.cap;
  // ---- bits shared by every key: no pass needed for them
  uint32_t k_and = 0xffffffffu, k_or = 0u;
  for (int i = ln; i < mycnt; i += 32) {
    k_and &= kb[i];
    k_or |= kb[i];
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    k_and &= __shfl_xor_sync(0xffffffffu, k_and, o);
    k_or |= __shfl_xor_sync(0xffffffffu, k_or, o);
  }
  if (t == 0) {
    s.all_and = 0xffffffffu;
    s.all_or = 0u;
  }
  e.sync();
  if (ln == 0 && mycnt > 0) {
    atomicAnd(&s.all_and, k_and);
    atomicOr(&s.all_or, k_or);
  }
  e.sync();
  const uint32_t diff = s.all_and ^ s.all_or;
  // ---- the k-th best key: MSB-first radix over the bits where keys differ
  int hi = diff ? 31 - __clz(diff) : -1;
  uint32_t mask = hi >= 0 ? ~((2u << hi) - 1u) : 0xffffffffu;  // (2u << 31) wraps to 0: all bits differ
  if (hi == 31) mask = 0u;
  uint32_t prefix = s.all_and & mask;
  int krem = k, n_tied = total;
#pragma unroll 1
  while (hi >= 0) {
    const int lo = hi >= 7 ? hi - 7 : 0;
    const uint32_t dmask = (hi - lo == 31) ? 0xffffffffu : ((1u << (hi - lo + 1)) - 1u);
    for (int i = t; i < 256; i += NT) s.hist[i] = 0;
    e.sync();
    for (int base = 0; base < mycnt; base += 32) {
      const int i = base + ln;
      const uint32_t key = i < mycnt ? kb[i] : 0u;
      warp_hist_add(s.hist, (i < mycnt && (key & mask) == prefix) ? (int)((key >> lo) & dmask) : -1);
    }
    e.sync();
    eng_pick_digit(e, krem, true);
    prefix |= static_cast<uint32_t>(s.sel_digit) << lo;
    mask |= dmask << lo;
    krem -= s.sel_before;
    n_tied = s.sel_count;
    hi = lo - 1;
  }
  const uint32_t thr = prefix;
  // ---- ties at thr: keep the krem lowest indices (indices are distinct)
  uint32_t jthr = 0xffffffffu;
  if (krem < n_tied) {
    uint32_t jp = 0u, jm = 0u;
    int jrem = krem;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = t; i < 256; i += NT) s.hist[i] = 0;
      e.sync();
      for (int base = 0; base < mycnt; base += 32) {
        const int i = base + ln;
        const bool in = i < mycnt;
        const uint32_t j = in ? static_cast<uint32_t>(jb[i]) : 0u;
        warp_hist_add(s.hist, (in && kb[i] == thr && (j & jm) == jp) ? (int)((j >> shift) & 255u) : -1);
      }
      e.sync();
      eng_pick_digit(e, jrem, false);
      jp |= static_cast<uint32_t>(s.sel_digit) << shift;
      jm |= 0xffu << shift;
      jrem -= s.sel_before;
    }
    jthr = jp;
  }
  // ---- compact every warp's buffer in place (writes never pass the read position)
  int wr = 0;
  for (int base = 0; base < mycnt; base += 32) {
    const int i = base + ln;
    const bool in = i < mycnt;
    const uint32_t key = in ? kb[i] : 0u;
    const int32_t j = in ? jb[i] : 0;
    const bool keep = in && (key > thr || (key == thr && static_cast<uint32_t>(j) <= jthr));
    const unsigned km = __ballot_sync(0xffffffffu, keep);
    if (keep) {
      const int o = wr + __popc(km & lanemask_lt());
      kb[o] = key;
      jb[o] = j;
    }
    wr += __popc(km);
    __syncwarp();
  }
  e.sync();
  if (ln == 0) s.warp_cnt[w] = wr;
  if (t == 0) s.thr = thr;
  e.sync();
}

// Shrinks the group's buffers with one histogram pass instead of eng_select's exact passes:
// over the 8 highest bits where the keys differ, the digit holding the k-th best key is found
// and every entry whose digit is below it is dropped (at least k entries lie at or above that
// digit's lower edge T, so every dropped entry ranks behind k others).  sh->thr becomes T, a
// valid append threshold (the exact k-th key is at least T).  Returns whether every buffer
// now has room for a round; when not (a crowded digit, or keys all equal) the caller selects
// exactly.  All threads of the group must call it.
template <int NW>
__device__ __noinline__ bool eng_prune(const Engine<NW> e, int k) {
  EngShared& s = *e.sh;
  const int t = e.tid, ln = e.lane(), w = e.warp();
  const int mycnt = s.warp_cnt[w];
  uint32_t* kb = e.keys + w * e.cap;
  int32_t* jb = e.js + w * e.cap;
  uint32_t k_and = 0xffffffffu, k_or = 0u;
  for (int i = ln; i < mycnt; i += 32) {
    k_and &= kb[i];
    k_or |= kb[i];
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    k_and &= __shfl_xor_sync(0xffffffffu, k_and, o);
    k_or |= __shfl_xor_sync(0xffffffffu, k_or, o);
  }
  if (t == 0) {
    s.all_and = 0xffffffffu;
    s.all_or = 0u;
  }
  for (int i = t; i < 256; i += NW * 32) s.hist[i] = 0;
  e.sync();
  if (ln == 0 && mycnt > 0) {
    atomicAnd(&s.all_and, k_and);
    atomicOr(&s.all_or, k_or);
  }
  e.sync();
  const uint32_t diff = s.all_and ^ s.all_or;
  if (diff == 0u) {  // every key equal: only the indices can decide
    e.sync();
    return false;
  }
  const int hi = 31 - __clz(diff), lo = hi >= 7 ? hi - 7 : 0;
  const uint32_t dmask = (1u << (hi - lo + 1)) - 1u;  // hi - lo <= 7
  for (int base = 0; base < mycnt; base += 32) {
    const int i = base + ln;
    warp_hist_add(s.hist, i < mycnt ? (int)((kb[i] >> lo) & dmask) : -1);
  }
  e.sync();
  eng_pick_digit(e, k, true);
  const uint32_t above = hi == 31 ? 0u : ~((2u << hi) - 1u);  // bits shared by every key
  const uint32_t T = (s.all_and & above) | (static_cast<uint32_t>(s.sel_digit) << lo);
  int wr = 0;
  for (int base = 0; base < mycnt; base += 32) {
    const int i = base + ln;
    const bool in = i < mycnt;
    const uint32_t key = in ? kb[i] : 0u;
    const int32_t j = in ? jb[i] : 0;
    const bool keep = in && key >= T;
    const unsigned km = __ballot_sync(0xffffffffu, keep);
    if (keep) {
      const int o = wr + __popc(km & lanemask_lt());
      kb[o] = key;
      jb[o] = j;
    }
    wr += __popc(km);
    __syncwarp();
  }
  e.sync();
  if (ln == 0) s.warp_cnt[w] = wr;
  if (t == 0) s.thr = max(s.thr, T);
  e.sync();
  bool room = true;
#pragma unroll
  for (int i = 0; i < NW; ++i) room &= s.warp_cnt[i] <= e.cap - kRoundEntries;
  e.sync();
  return room;
}

// eng_check that first tries the one-pass prune (eng_prune) when some buffer could overflow
// before the next check, and selects exactly only when that leaves too little room.  Returns
// the threshold and refreshes `cnt`.
template <int NW>
__device__ __forceinline__ uint32_t eng_check_fast(const Engine<NW>& e, int k, int& cnt) {
  if (e.lane() == 0) e.sh->warp_cnt[e.warp()] = cnt;
  e.sync();
  bool need = false;
#pragma unroll
  for (int i = 0; i < NW; ++i) need |= e.sh->warp_cnt[i] > e.cap - kRoundEntries;
  if (need && !eng_prune(e, k)) eng_select(e, k);  // uniform: every thread read the same counts
  cnt = e.sh->warp_cnt[e.warp()];
  const uint32_t thr = e.sh->thr;
  e.sync();
  return thr;
}

// Publishes the warp counts and selects when some buffer could overflow before the next
// check.  Returns the (possibly raised) threshold and refreshes `cnt`.
template <int NW>
__device__ __forceinline__ uint32_t eng_check(const Engine<NW>& e, int k, int& cnt) {
  if (e.lane() == 0) e.sh->warp_cnt[e.warp()] = cnt;
  e.sync();
  bool need = false;
#pragma unroll
  for (int i = 0; i < NW; ++i) need |= e.sh->warp_cnt[i] > e.cap - kRoundEntries;
  if (need) eng_select(e, k);  // uniform: every thread read the same counts
  cnt = e.sh->warp_cnt[e.warp()];
  const uint32_t thr = e.sh->thr;
  e.sync();
  return thr;
}

// Places the survivors of a select, sorted by entry index, in out_key / out_j [0..n) and
// returns n.  *thr_out gets the k-th key when k survive, else 0 (every dropped entry has a
// key <= it, and the row's k-th key is at least it).
template <int NW>
__device__ int eng_rank(const Engine<NW>& e, int k, uint32_t* thr_out) {
  int total = 0;
#pragma unroll
  for (int i = 0; i < NW; ++i) total += e.sh->warp_cnt[i];
  // Every warp's buffer is in ascending entry order (appends arrive in order and compaction
  // keeps it), so an entry's rank among all survivors is its index in its own buffer plus,
  // for every other warp, the number of that warp's survivors with a smaller index.
  const int w = e.warp();
  const int mycnt = e.sh->warp_cnt[w];
  const uint32_t* gk = e.keys + w * e.cap;
  const int32_t* gj = e.js + w * e.cap;
  for (int i = e.lane(); i < mycnt; i += 32) {
    const int32_t ji = gj[i];
    int r = i;
#pragma unroll 1
    for (int w2 = 0; w2 < NW; ++w2) {
      if (w2 == w) continue;
      const int32_t* bj = e.js + w2 * e.cap;
      int lo2 = 0, hi2 = e.sh->warp_cnt[w2];
      while (lo2 < hi2) {
        const int mid = (lo2 + hi2) >> 1;
        if (bj[mid] < ji) lo2 = mid + 1; else hi2 = mid;
      }
      r += lo2;
    }
    e.out_key[r] = gk[i];
    e.out_j[r] = ji;
  }
  if (e.tid == 0 && thr_out) *thr_out = total >= k ? e.sh->thr : 0u;
  e.sync();
  return total;
}

// Final select, then eng_rank.  k <= kEngMaxK.
template <int NW>
__device__ int eng_finish(const Engine<NW>& e, int k, int cnt, uint32_t* thr_out) {
  if (e.lane() == 0) e.sh->warp_cnt[e.warp()] = cnt;
  e.sync();
  eng_select(e, k);
  return eng_rank(e, k, thr_out);
}

// Balanced split of [0, n) into `parts` contiguous ranges; range `i`.
__device__ __forceinline__ void split_range(long long n, int parts, int i, long long& lo, long long& hi) {
  lo = (n * i) / parts;
  hi = (n * (i + 1)) / parts;
}

}  // namespace csa2
