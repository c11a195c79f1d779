// Exact streaming top-K for one row per thread block (512 threads = 16 warps).
//
// Selection rule ("06 / Indexer and attention", select_values, and its note that ties use
// the lower position first): keep the K entries that are best by (score descending, entry
// order ascending).  Scores are compared through order-preserving uint32 keys
// (score_key), so -0.0 == +0.0 and the comparison is exact.
//
// State: every warp owns a buffer of (key, position) pairs holding ITS surviving entries in
// entry order; warps own consecutive entry ranges in warp order, so the concatenation of
// the buffers is in entry order.  A warp appends survivors of each 32-entry group with a
// ballot (order preserved).  An entry survives if its key exceeds `thr`, the K-th best key
// seen so far (0 until K entries have been seen): a later entry with a key <= thr ranks
// behind at least K earlier entries and can never be selected.  When a buffer nears its
// capacity the block runs `engine_select`: an MSB-first 8-bit radix select finds the K-th
// key and how many entries equal to it to keep, then every warp compacts its buffer in
// place.  The result after the last select is exactly the top-K, in entry order.
#pragma once

#include "common.cuh"

namespace csa2 {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kRoundEntries = 128;  // most entries one warp appends between two checks

struct SelectShared {
  int hist[256];
  int tmp[32];
  int warp_cnt[kSelWarps];
  int warp_eq[kSelWarps];
  uint32_t thr;
  int sel_digit;
  int sel_above;
  int total;
};

struct TopkEngine {
  uint32_t* keys;  // [kSelWarps * cap]
  int32_t* pos;    // [kSelWarps * cap]
  int cap;         // per-warp capacity, >= K + kRoundEntries
  SelectShared* sh;
};

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ void engine_init(TopkEngine& e) {
  if (threadIdx.x < kSelWarps) e.sh->warp_cnt[threadIdx.x] = 0;
  if (threadIdx.x == 0) e.sh->thr = 0u;
  __syncthreads();
}

// Appends, in lane order, the lanes' entries that are valid and beat `thr`.  `cnt` is the
// warp's buffer fill (warp-uniform register).  The caller guarantees room for 32 more.
__device__ __forceinline__ void warp_append(const TopkEngine& e, int wid, int& cnt, uint32_t thr,
                                            bool valid, uint32_t key, int32_t pos) {
  const bool keep = valid && key > thr;
  const unsigned m = __ballot_sync(0xffffffffu, keep);
  if (keep) {
    const int o = wid * e.cap + cnt + __popc(m & lanemask_lt());
    e.keys[o] = key;
    e.pos[o] = pos;
  }
  cnt += __popc(m);
}

// Block-wide: keep the top-k of the concatenated warp buffers (counts in sh->warp_cnt).
// Updates sh->warp_cnt and sh->thr.  Must be called by all threads.
__device__ inline void engine_select(const TopkEngine& e, int k) {
  SelectShared& s = *e.sh;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int mycnt = s.warp_cnt[wid];
  int total = 0;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) total += s.warp_cnt[w];
  if (total <= k) {
    __syncthreads();
    return;
  }
  const uint32_t* kb = e.keys + wid * e.cap;
  int32_t* pb = e.pos + wid * e.cap;
  uint32_t prefix = 0u, mask = 0u;
  int krem = k;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    if (tid < 256) s.hist[tid] = 0;
    __syncthreads();
    for (int i = lane; i < mycnt; i += 32) {
      const uint32_t key = kb[i];
      if ((key & mask) == prefix) atomicAdd(&s.hist[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    const int c = tid < 256 ? s.hist[255 - tid] : 0;
    int tot;
    const int above = block_excl_scan<kSelThreads>(c, s.tmp, &tot);  // entries with a larger digit
    if (tid < 256 && above < krem && above + c >= krem) {
      s.sel_digit = 255 - tid;
      s.sel_above = above;
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(s.sel_digit) << shift;
    mask |= 0xffu << shift;
    krem -= s.sel_above;
  }
  const uint32_t thr = prefix;  // the k-th best key
  const int n_eq = krem;        // entries equal to thr to keep, first ones in entry order

  int eq = 0;
  for (int i = lane; i < mycnt; i += 32) eq += (kb[i] == thr);
#pragma unroll
  for (int o = 16; o; o >>= 1) eq += __shfl_xor_sync(0xffffffffu, eq, o);
  if (lane == 0) s.warp_eq[wid] = eq;
  __syncthreads();
  int eq_before = 0;
  for (int w = 0; w < wid; ++w) eq_before += s.warp_eq[w];
  const int take = max(0, min(eq, n_eq - eq_before));

  int wr = 0, eq_seen = 0;
  uint32_t* kw = e.keys + wid * e.cap;
  for (int base = 0; base < mycnt; base += 32) {
    const int i = base + lane;
    const bool in = i < mycnt;
    const uint32_t key = in ? kw[i] : 0u;
    const int32_t p = in ? pb[i] : 0;
    const bool is_eq = in && key == thr;
    const unsigned em = __ballot_sync(0xffffffffu, is_eq);
    const int eq_rank = eq_seen + __popc(em & lanemask_lt());
    const bool keep = in && (key > thr || (is_eq && eq_rank < take));
    const unsigned km = __ballot_sync(0xffffffffu, keep);
    if (keep) {
      const int o = wr + __popc(km & lanemask_lt());
      kw[o] = key;
      pb[o] = p;
    }
    wr += __popc(km);
    eq_seen += __popc(em);
    __syncwarp();
  }
  __syncthreads();
  if (lane == 0) s.warp_cnt[wid] = wr;
  if (tid == 0) s.thr = thr;
  __syncthreads();
}

// Publishes the warp counts and selects when some buffer could overflow in the next round.
// Returns the (possibly raised) threshold; `cnt` is refreshed.  All threads must call it.
__device__ __forceinline__ uint32_t engine_round_end(const TopkEngine& e, int k, int wid, int lane,
                                                     int& cnt) {
  if (lane == 0) e.sh->warp_cnt[wid] = cnt;
  __syncthreads();
  bool need = false;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) need |= e.sh->warp_cnt[w] > e.cap - kRoundEntries;
  if (need) engine_select(e, k);  // uniform branch: every thread read the same counts
  cnt = e.sh->warp_cnt[wid];
  const uint32_t thr = e.sh->thr;
  __syncthreads();
  return thr;
}

// Final select, then writes the kept entries in entry order.  With `final_idx`, writes
// positions to final_idx[0..k) padded with -1; otherwise writes keys/positions to
// out_keys/out_pos[0..n) and n to *out_cnt.
__device__ inline void engine_finish(const TopkEngine& e, int k, int wid, int lane, int cnt, int32_t* final_idx,
                              uint32_t* out_keys, int32_t* out_pos, int32_t* out_cnt) {
  if (lane == 0) e.sh->warp_cnt[wid] = cnt;
  __syncthreads();
  engine_select(e, k);
  const int mycnt = e.sh->warp_cnt[wid];
  int off = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) {
    const int c = e.sh->warp_cnt[w];
    off += (w < wid) ? c : 0;
    total += c;
  }
  const uint32_t* kb = e.keys + wid * e.cap;
  const int32_t* pb = e.pos + wid * e.cap;
  if (final_idx) {
    for (int i = lane; i < mycnt; i += 32) final_idx[off + i] = pb[i];
    for (int i = total + threadIdx.x; i < k; i += kSelThreads) final_idx[i] = -1;
  } else {
    for (int i = lane; i < mycnt; i += 32) {
      out_keys[off + i] = kb[i];
      out_pos[off + i] = pb[i];
    }
    if (threadIdx.x == 0) *out_cnt = total;
  }
}

// Balanced split of [0, n) into `parts` contiguous ranges; range `i`.
__device__ __forceinline__ void split_range(long long n, int parts, int i, long long& lo, long long& hi) {
  lo = (n * i) / parts;
  hi = (n * (i + 1)) / parts;
}

}  // namespace csa2
