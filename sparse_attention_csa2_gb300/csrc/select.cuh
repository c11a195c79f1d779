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
// `eng_finish` emits the survivors sorted by index (rank counting).
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
};

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Histogram increment aggregated over the warp: lanes with equal bins add once (scores of a
// row share their leading key bits, so plain per-lane atomics would serialise on one bin).
// `bin` < 0 adds nothing.  All lanes of the warp must call it.
__device__ __forceinline__ void warp_hist_add(int* hist, int bin) {
  const unsigned act = __ballot_sync(0xffffffffu, bin >= 0);
  if (bin >= 0) {
    const unsigned peers = __match_any_sync(act, bin);
    if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
  }
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
  // ---- the k-th best key: MSB-first radix over the keys
  uint32_t prefix = 0u, mask = 0u;
  int krem = k, n_tied = 0;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = t; i < 256; i += NT) s.hist[i] = 0;
    e.sync();
    for (int base = 0; base < mycnt; base += 32) {
      const int i = base + ln;
      const uint32_t key = i < mycnt ? kb[i] : 0u;
      warp_hist_add(s.hist, (i < mycnt && (key & mask) == prefix) ? (int)((key >> shift) & 255u) : -1);
    }
    e.sync();
    eng_pick_digit(e, krem, true);
    prefix |= static_cast<uint32_t>(s.sel_digit) << shift;
    mask |= 0xffu << shift;
    krem -= s.sel_before;
    n_tied = s.sel_count;
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

// Final select; the survivors, sorted by entry index, go to out_key / out_j [0..n) and n is
// returned.  *thr_out gets the k-th key when k survive, else 0 (every dropped entry has a
// key <= it, and the row's k-th key is at least it).  k <= kEngMaxK.
template <int NW>
__device__ int eng_finish(const Engine<NW>& e, int k, int cnt, uint32_t* thr_out) {
  constexpr int NT = NW * 32;
  constexpr int PER = (kEngMaxK + NT - 1) / NT;
  if (e.lane() == 0) e.sh->warp_cnt[e.warp()] = cnt;
  e.sync();
  eng_select(e, k);
  int off = 0, total = 0;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    const int c = e.sh->warp_cnt[i];
    off += (i < e.warp()) ? c : 0;
    total += c;
  }
  const int mycnt = e.sh->warp_cnt[e.warp()];
  const uint32_t* gk = e.keys + e.warp() * e.cap;
  const int32_t* gj = e.js + e.warp() * e.cap;
  for (int i = e.lane(); i < mycnt; i += 32) {
    e.out_key[off + i] = gk[i];
    e.out_j[off + i] = gj[i];
  }
  e.sync();
  // rank of an entry = number of survivors with a smaller index
  uint32_t mk[PER];
  int32_t mj[PER], mr[PER];
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int i = e.tid + q * NT;
    mr[q] = -1;
    if (i < total) {
      mk[q] = e.out_key[i];
      mj[q] = e.out_j[i];
      int r = 0;
      for (int m = 0; m < total; ++m) r += e.out_j[m] < mj[q];
      mr[q] = r;
    }
  }
  e.sync();
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    if (mr[q] >= 0) {
      e.out_key[mr[q]] = mk[q];
      e.out_j[mr[q]] = mj[q];
    }
  }
  if (e.tid == 0 && thr_out) *thr_out = total >= k ? e.sh->thr : 0u;
  e.sync();
  return total;
}

// Balanced split of [0, n) into `parts` contiguous ranges; range `i`.
__device__ __forceinline__ void split_range(long long n, int parts, int i, long long& lo, long long& hi) {
  lo = (n * i) / parts;
  hi = (n * (i + 1)) / parts;
}

}  // namespace csa2
