// Lightning indexer on the 5th-generation tensor cores (tcgen05, TMA, tensor memory).
//
// score_j = sum_h w_h * ReLU(q^I_h . k^I_j) ("Every layer, connected", "The global and index
// paths") as one dense contraction per 128-record tile:
//   D[128 records x 32*NQ] = K_tile[128 x 128] * Q[32*NQ x 128]^T      (bf16 in, fp32 in TMEM)
// with the records along M (TMEM lanes) and (query, head) along N (TMEM columns), so that
// every epilogue thread owns one record and reads its 32 head dot products per query with a
// single tcgen05.ld, then applies ReLU, the head weights and the head sum in registers.
//
// Roles (one thread block): warp 0 issues TMA tile loads into a ring of shared-memory stages,
// warp 1 allocates tensor memory and one of its threads issues the MMAs, and the epilogue
// warps drain the double-buffered accumulators.  Every mbarrier wait is bounded: on a
// timeout the block records CSA2_ETIMEOUT, finishes its loops without waiting, drains what it
// issued (bounded again), frees its tensor memory and returns.
//
//   decode  (NQ = 1): one query row per block, one contiguous segment of its visible records;
//                     the epilogue feeds the exact top-K engine and the block maxima.
//   prefill (NQ = 8): a persistent grid walks (8-query tile, key range) work items of one
//                     sequence; causal masking per query; scores are written out.
#include <cudaTypedefs.h>
#include <mutex>

#include "kernels.h"
#include "array_topk.cuh"
#include "select.cuh"
#include "tc05.cuh"

namespace csa2 {
namespace {

constexpr int kTileKeys = 128;
constexpr int kKeyHalf = kTileKeys * 128;   // one K-half (64 dims) of a key tile: 16 KB
constexpr int kKeyTile = 2 * kKeyHalf;      // 32 KB

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ void report_timeout(int* flag, int32_t* dev_status) {
  *flag = 1;
  if (dev_status != nullptr) atomicExch(dev_status, (int)CSA2_ETIMEOUT);
}

// E4M3 terms of q^I for the FP8 decode scans (construction in the comment below): thread et
// (0..255) takes head et / 8, dims 16 (et % 8) .. +15, and writes its three terms into the B
// operand qs (row 32 * term + head, 128 bytes per row, 128-byte swizzle); the thread with
// et % 8 == 0 stores the head's power-of-two exponent in qexp[head].
__device__ __forceinline__ void fp8_q_terms(const void* q_idx, int row, int et, uint8_t* qs, int* qexp) {
  const int h = et >> 3, c = et & 7;
  const uint4* src = reinterpret_cast<const uint4*>(q_idx) + ((size_t)row * 32 + h) * 16 + 2 * c;
  const uint4 u0 = __ldg(src), u1 = __ldg(src + 1);
  const uint32_t qw[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
  uint32_t mx = 0u;
#pragma unroll
  for (int k = 0; k < 8; ++k) mx = max(mx, max(qw[k] & 0x7fffu, (qw[k] >> 16) & 0x7fffu));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  // largest magnitude 2^ex * m, m in [1, 2): scale by 2^(7 - ex) into [128, 256)
  const int ex = (int)((mx >> 7) & 0xffu) - 127;
  const int e = mx == 0u ? 0 : min(126, max(-126, 7 - ex));
  const float f = __int_as_float((e + 127) << 23);
  uint32_t term[3][4];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    float x[2] = {__uint_as_float(qw[k] << 16) * f, __uint_as_float(qw[k] & 0xffff0000u) * f};
#pragma unroll
    for (int tm = 0; tm < 3; ++tm) {
      const uint16_t b2 = __nv_cvt_float2_to_fp8x2(make_float2(x[0], x[1]), __NV_SATFINITE, __NV_E4M3);
      const uint32_t hb = e4m3x2_to_f16x2(b2);
      const float2 back = __half22float2(*reinterpret_cast<const __half2*>(&hb));
      x[0] = (x[0] - back.x) * 16.f;  // exact: the residual has at most 4 significant bits
      x[1] = (x[1] - back.y) * 16.f;
      if (k & 1) term[tm][k >> 1] |= (uint32_t)b2 << 16;
      else term[tm][k >> 1] = b2;
    }
  }
#pragma unroll
  for (int tm = 0; tm < 3; ++tm) {
    const int n = 32 * tm + h;  // B row; 16-byte chunk c sits at slot c ^ (n & 7)
    *reinterpret_cast<uint4*>(qs + n * 128 + ((c ^ (n & 7)) << 4)) =
        make_uint4(term[tm][0], term[tm][1], term[tm][2], term[tm][3]);
  }
  if (c == 0) qexp[h] = e;
}

// ===================================================================================== decode
// bf16 keys: TMA tiles of 128 records x 256 bytes; D[128 x 32] += K_tile * Q^T in eight
// kind::f16 K-steps of 16.
// FP8 keys (E4M3 with one fp32 scale per record): TMA tiles of 128 records x 128 bytes used as
// they are, in four kind::f8f6f4 K-steps of 32.  q^I (bf16) becomes three E4M3 terms per
// element: each head is scaled by the power of two that puts its largest element in
// [128, 256), then x = t1 + t2 / 16 + t3 / 256 with t1 = rn(x), t2 = rn(16 (x - t1)),
// t3 = rn(16 (16 (x - t1) - t2)), every residual exact in fp32.  Two terms already hold any
// element whose exponent is at least 2^-6 (8 significant bits against E4M3's 4); the third
// carries smaller ones down to 2^-10 exactly, that is every element within 2^-17 of its
// head's largest.  B is the [96 x 128] E4M3 matrix of the terms (row 32 * term + head), D
// the [128 x 96] products, and the epilogue sums D1 + D2 / 16 + D3 / 256 per head, takes the
// record's scale, then ReLU and the head weight (times the inverse power of two).
template <bool FP8>
struct DecCfg {
  static constexpr int kStages = FP8 ? 8 : 4;
  static constexpr int kTileBytes = FP8 ? kTileKeys * 128 : kKeyTile;
  static constexpr int kThreads = 12 * 32;  // warp 0 TMA, warp 1 MMA + TMEM, warps 4..11 epilogue
  static constexpr int kQBytes = FP8 ? 96 * 128 : 2 * 32 * 128;  // E4M3 terms, or the bf16 query tile
  static constexpr int kN = FP8 ? 96 : 32;                         // MMA N
  static constexpr uint32_t kAccCols = FP8 ? 128 : 32;             // columns per accumulator
  static constexpr uint32_t kTmemCols = FP8 ? 256 : 64;
  static_assert(kStages * kTileBytes == 4 * kKeyTile, "both rings have the same size");
};
constexpr int kDecRingBytes = 4 * kKeyTile;
constexpr int kDecEpiFirst = 4;
constexpr int kDecEpiWarps = 8;  // two groups of 4 warps (one per TMEM lane quarter), alternate tiles
constexpr int kDecQHalf = 32 * 128;  // bf16: 32 heads x 64 dims x 2 B
constexpr int kDecSegMax = 16384;    // records of one segment (their keys stay in shared memory)
// Cluster selection with marked candidates: at most this many marked entries per row (their
// keys and positions, then the selection's lists, fit in the idle tile ring), and the bytes of
// the per-segment bitmap of marked entries.
constexpr int kFastCap = 6144;
constexpr int kFastBytes = kDecSegMax / 8;
constexpr int kMaxClusterSeg = 16;

struct DecBars {
  uint64_t full[8], empty[8], tfull[2], tempty[2], qfull, qready;
  uint32_t tmem_base;
  int timeout;
  int issued;     // tiles whose TMA loads were issued
  int consumed;   // tiles whose MMAs were issued
  int drained;    // tiles whose accumulators the epilogue read
  int last;       // this block is the last segment of its row to finish
  int qexp[32];   // FP8: power-of-two exponent applied to each head of q^I
  // marked-candidate selection
  int tile_keys[16];   // per tile slot (t mod 16): epilogue warps that stored tile t's keys
  uint32_t maxkey;     // largest key the lister has seen (read by the other blocks' listers)
  int lister_fail;     // the lister's wait gave up
  int cand_cnt[kMaxClusterSeg];      // per block: its marked entries (-1: not usable), pushed by it
  uint32_t cand_lo[kMaxClusterSeg];  // per block: its lister's last bound (<= the row's K-th key)
  uint32_t cand_hi[kMaxClusterSeg];  // per block: the largest key of its segment
  uint32_t bound;                    // this block's lister's last bound
  int cand_off[kMaxClusterSeg + 1];  // per block: offset of its entries in the row's list; [n] = total
  int cand_go;         // the row's marked entries fit: block 0 selects among them
};

// The last segment block of a row merges the row's lists: every list entry's key goes into
// the key array (entries below the largest per-segment K-th key cannot be selected and are
// left out, and the level-1 histogram is counted on the way), and the K best, in position
// order, become the row's indices.  The lists (and, with room in the scratch, their
// positions) come into shared memory in one batch of asynchronous copies, so the merge waits
// for the L2 only once.
template <int NW>
__device__ void merge_row_lists(const ArrSel<NW>& sel, uint32_t* keys, const ScanParams& p, int row, int n_seg,
                                int32_t* sel_idx, int list_room) {
  constexpr int NT = NW * 32;
  const int K = p.K, n = n_seg * K;
  const uint32_t* lists = p.seg_keys + (size_t)row * n_seg * K;
  const int32_t* pos = p.seg_pos + (size_t)row * n_seg * K;
  const int lw = ArrSel<NW>::list_words(n);
  int32_t* pos_s = lw + n <= list_room ? reinterpret_cast<int32_t*>(sel.scratch + lw) : nullptr;
  const bool vec = (K & 3) == 0 && ((reinterpret_cast<uintptr_t>(p.seg_keys) | reinterpret_cast<uintptr_t>(p.seg_pos)) & 15) == 0;
  if (vec) {
    for (int c = sel.tid; c < n / 4; c += NT) {
      cp_async16(keys + 4 * c, lists + 4 * c, true);
      if (pos_s) cp_async16(pos_s + 4 * c, pos + 4 * c, true);
    }
    cp_async_commit();
  } else {
    pos_s = nullptr;
    for (int f = sel.tid; f < n; f += NT) keys[f] = __ldcg(lists + f);
  }
  // segment counts and K-th keys staged in shared memory (n_seg <= 64)
  int* cnt_s = reinterpret_cast<int*>(sel.sh->aux);
  uint32_t* thr_s = sel.sh->aux + 64;
  for (int s = sel.tid; s < n_seg; s += NT) {
    cnt_s[s] = __ldcg(p.seg_cnt + (size_t)row * n_seg + s);
    thr_s[s] = __ldcg(p.seg_thr + (size_t)row * n_seg + s);
  }
  sel.zero_hist(kHistBins);
  cp_async_wait<0>();
  sel.sync();
  uint32_t thr0 = 0u;
  for (int s = 0; s < n_seg; ++s) thr0 = max(thr0, thr_s[s]);
  // unused list slots and keys below thr0 leave the candidates
  for (int sg = 0; sg < n_seg; ++sg) {
    const int cnt = cnt_s[sg];
    for (int j = sel.tid; j < K; j += NT) {
      uint32_t key = keys[sg * K + j];
      if (j >= cnt || key < thr0) key = 0u;
      keys[sg * K + j] = key;
      hist_add(sel.sh->hist, key >> 20, key != 0u);
    }
  }
  sel.sync();
  arr_threshold(sel, keys, n, K, true);
  const int kept = arr_compact(sel, n, sel_idx);
  int32_t* out = p.idx + (size_t)row * K;
  for (int r = sel.tid; r < K; r += NT) out[r] = r < kept ? (pos_s ? pos_s[sel_idx[r]] : __ldcg(pos + sel_idx[r])) : -1;
}

// ---- marked-candidate selection (the segments of a row form a cluster)
//
// While the tiles stream, one otherwise idle warp of every segment block (the lister) follows
// the epilogue tile by tile.  After half and after three quarters of its tiles it derives a lower
// bound on the row's K-th key from the level-1 histograms of all blocks of the cluster: the
// highest bin whose count from the top reaches K.  The counts only grow and each counts keys
// that exist, so however stale a remote read is, at least K keys of the row lie at or above
// that bin's lower edge, and so does the row's K-th key.  The lister marks, in a bitmap of its
// segment, every key at or above its latest bound (the tiles before the first bound once it
// exists); every selected entry of the row is therefore marked.  After the stream each block
// compacts its marked entries, and one block selects the row's top-K among all of them.

// Waits until the four epilogue warps that drain tile t have stored its keys (a per-slot
// count that grows by four per tile of the slot).  Bounded; false when it gave up.
__device__ __forceinline__ bool wait_tile_keys(const int* tile_keys, int t) {
  const int need = 4 * (t / 16 + 1);
  const volatile int* c = tile_keys + (t & 15);
  for (uint32_t i = 0; i < tc05::kSpinLimit; ++i) {
    if (*c >= need) {
      __threadfence_block();
      return true;
    }
    __nanosleep(32);
  }
  return false;
}

// Lower bound on the row's K-th key from the cluster's level-1 histograms (key >> 20), read
// from the top: blocks publish the largest key they have seen, the warp sums 128 bins of every
// block per step (lane l: the four bins hi - 4l - 3 .. hi - 4l) until the count from the top
// reaches K.  Returns that bin's lower edge, or 0 while fewer than K keys are counted.
__device__ __forceinline__ uint32_t row_key_bound(const int* hist, const uint32_t* maxkey, uint32_t n_cta, int K) {
  const int lane = threadIdx.x & 31;
  uint32_t top = 0u;
  if ((uint32_t)lane < n_cta) top = (uint32_t)cluster_ld_s32(cluster_map(maxkey, (uint32_t)lane));
#pragma unroll
  for (int o = 16; o; o >>= 1) top = max(top, __shfl_xor_sync(0xffffffffu, top, o));
  if (top == 0u) return 0u;
  int cum = 0;
#pragma unroll 1
  for (int hi = (int)(top >> 20) | 3; hi >= 3; hi -= 128) {
    const int b0 = hi - 4 * lane - 3;  // a multiple of 4
    int s0 = 0, s1 = 0, s2 = 0, s3 = 0;
    if (b0 >= 0) {
      // every block's four bins at once: the remote loads' round trips overlap (one after
      // another they cost ~2 us per bound at 8 blocks)
      uint4 v[kMaxClusterSeg];
#pragma unroll
      for (int r = 0; r < kMaxClusterSeg; ++r)
        if ((uint32_t)r < n_cta) v[r] = cluster_ld_v4(cluster_map(hist + b0, (uint32_t)r));
#pragma unroll
      for (int r = 0; r < kMaxClusterSeg; ++r)
        if ((uint32_t)r < n_cta) {
          s0 += (int)v[r].x;
          s1 += (int)v[r].y;
          s2 += (int)v[r].z;
          s3 += (int)v[r].w;
        }
    }
    const int c = s0 + s1 + s2 + s3;
    int inc = c;  // lanes in order = bins from the top down
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    const int tot = __shfl_sync(0xffffffffu, inc, 31);
    if (cum + tot >= K) {
      const unsigned m = __ballot_sync(0xffffffffu, cum + inc >= K);
      const int L = __ffs(m) - 1;
      int bin = b0;
      const int acc = cum + inc - c;
      if (acc + s3 >= K) bin = b0 + 3;
      else if (acc + s3 + s2 >= K) bin = b0 + 2;
      else if (acc + s3 + s2 + s1 >= K) bin = b0 + 1;
      bin = __shfl_sync(0xffffffffu, bin, L);
      return (uint32_t)bin << 20;
    }
    cum += tot;
  }
  return 0u;
}

// Marks tile t's keys at or above `bound` (lane l: keys 32u + l of the tile, u = 0..3; word
// 4t + u of the bitmap holds keys 32u .. 32u + 31).
__device__ __forceinline__ void mark_tile(uint32_t* listed, const uint32_t* keys, int t, int seg_len, uint32_t bound) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int j = t * kTileKeys + 32 * u + lane;
    const uint32_t k = j < seg_len ? keys[j] : 0u;
    const unsigned m = __ballot_sync(0xffffffffu, k != 0u && k >= bound);
    if (lane == u) listed[4 * t + u] = m;
  }
}

// Exact top-K among n marked entries (keys ck[0..n), record positions cp[0..n) in position
// order; n <= kFastCap), written to out[0..K) as ascending positions, -1 padded.  The caller
// gives lo <= the K-th key and hi >= every key (the listers' bounds and maxima) and has zeroed
// sh.hist and sh.aux.  One histogram of (key - lo) >> shift over 4096 bins (shift the smallest
// that fits [lo, hi]) with a coarse copy of 64 bins finds, in one warp, the bin of the K-th key
// and the count above it; the few keys of that bin go to one warp, which finds the K-th key T
// and how many entries equal to T are kept (the lowest positions first) by counting; a bin of
// more than 32 keys (ties) takes further histogram levels instead.  Each thread then takes a
// contiguous run of entries and one block scan places the selected ones.
template <int NW>
__device__ __noinline__ void select_marked(const ArrSel<NW>& s, const uint32_t* ck, const int32_t* cp, int n, int K,
                                           uint32_t lo, uint32_t hi, int32_t* out) {
  constexpr int NT = NW * 32;
  ArrSelShared& sh = *s.sh;
  const int tid = s.tid, lane = tid & 31;
  int* coarse = reinterpret_cast<int*>(sh.aux);        // 64 bins of 64 bins
  uint32_t* few = sh.aux + 64;                          // the keys of the K-th key's bin (<= 32)
  int* few_n = reinterpret_cast<int*>(sh.aux + 96);
  const int c = (n + NT - 1) / NT;
  const int a0 = min(n, tid * c), a1 = min(n, a0 + c);
  uint32_t thr = 0u;
  int n_eq = 0;
  if (n > K) {
    const int width = 32 - __clz(max(hi - lo, 1u));
    const int shift = max(0, width - 12);
#pragma unroll 2
    for (int i = a0; i < a1; ++i)
      if (ck[i] >= lo) {
        const uint32_t f = (ck[i] - lo) >> shift;
        atomicAdd(&sh.hist[f], 1);
        atomicAdd(&coarse[f >> 6], 1);
      }
    s.sync();
    if (s.warp() == 0) {
      // from the top: the coarse bin where the count reaches K, then its fine bin
      int above = 0, bin = 0;
#pragma unroll 1
      for (int stage = 0; stage < 2; ++stage) {
        const int* h = stage == 0 ? coarse : sh.hist + 64 * bin;
        const int x0 = h[63 - 2 * lane], x1 = h[62 - 2 * lane];
        int inc = x0 + x1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += y;
        }
        const int L = __ffs(__ballot_sync(0xffffffffu, above + inc >= K)) - 1;
        const int acc = above + inc - (x0 + x1);
        const int hit = acc + x0 >= K ? 63 - 2 * lane : 62 - 2 * lane;
        const int acc2 = acc + x0 >= K ? acc : acc + x0;
        const int b2 = __shfl_sync(0xffffffffu, hit, L);
        above = __shfl_sync(0xffffffffu, acc2, L);
        bin = stage == 0 ? b2 : 64 * bin + b2;
      }
      if (lane == 0) {
        sh.bin = bin;
        sh.before = above;
      }
    }
    s.sync();
    int need = K - sh.before;
    uint32_t base = lo + ((uint32_t)sh.bin << shift);
    if (shift == 0) {
      thr = base;
      n_eq = need;
    } else {
      const uint64_t top = (uint64_t)base + (1ull << shift);
#pragma unroll 2
      for (int i = a0; i < a1; ++i)
        if (ck[i] >= base && (uint64_t)ck[i] < top) {
          const int slot = atomicAdd(few_n, 1);
          if (slot < 32) few[slot] = ck[i];
        }
      s.sync();
      const int p = *few_n;
      if (p <= 32) {
        if (s.warp() == 0) {
          // the need-th largest of the bin's keys, by counting
          const uint32_t x = lane < p ? few[lane] : 0u;
          int gt = 0, ge = 0;
#pragma unroll 1
          for (int j = 0; j < p; ++j) {
            const uint32_t y = __shfl_sync(0xffffffffu, x, j);
            gt += y > x;
            ge += y >= x;
          }
          const unsigned m = __ballot_sync(0xffffffffu, lane < p && gt < need && need <= ge);
          const int L = __ffs(m) - 1;
          if (lane == L) {
            sh.thr = x;
            sh.n_eq = need - gt;
          }
        }
        s.sync();
        thr = sh.thr;
        n_eq = sh.n_eq;
      } else {
        // many keys in the bin (ties): 4096-bin levels over it until the bins are single keys
        int width2 = shift;
#pragma unroll 1
        while (true) {
          const int sh2 = max(0, width2 - 12);
          s.sync();
          for (int i = tid; i < kHistBins; i += NT) sh.hist[i] = 0;
          s.sync();
          const uint64_t top2 = (uint64_t)base + (1ull << width2);
#pragma unroll 2
          for (int i = a0; i < a1; ++i)
            if (ck[i] >= base && (uint64_t)ck[i] < top2) atomicAdd(&sh.hist[(ck[i] - base) >> sh2], 1);
          s.sync();
          s.template pick<kHistBins>(need);
          need -= sh.before;
          base += (uint32_t)sh.bin << sh2;
          if (sh2 == 0) break;
          width2 = sh2;
        }
        thr = base;
        n_eq = need;
      }
    }
  }
  // compaction: the thread's run of entries, placed by one block scan
  int gt = 0, eq = 0;
  if (n <= K) {
    gt = a1 - a0;
  } else {
#pragma unroll 2
    for (int i = a0; i < a1; ++i) {
      gt += ck[i] > thr;
      eq += ck[i] == thr;
    }
  }
  int tot;
  const int before = s.scan((gt << 16) | eq, &tot);
  const int eq_b = before & 0xffff;
  int at = (before >> 16) + min(eq_b, n_eq);
  int take = max(0, min(eq, n_eq - eq_b));
#pragma unroll 2
  for (int i = a0; i < a1; ++i) {
    const uint32_t k = ck[i];
    bool keep = n <= K || k > thr;
    if (!keep && k == thr && take > 0) {
      keep = true;
      --take;
    }
    if (keep) out[at++] = cp[i];
  }
  const int kept = (tot >> 16) + min(tot & 0xffff, n_eq);
  for (int r = kept + tid; r < K; r += NT) out[r] = -1;
}

template <bool FP8>
__global__ void __launch_bounds__(DecCfg<FP8>::kThreads, 1)
    idx_mma_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                          const __grid_constant__ CUtensorMap tmK64, const ScanParams p) {
  using C = DecCfg<FP8>;
  constexpr int kStages = C::kStages, kThreads = C::kThreads;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* ring = smem;
  uint8_t* qs = ring + kDecRingBytes;
  DecBars& bars = *reinterpret_cast<DecBars*>(qs + C::kQBytes);
  uint8_t* rest = reinterpret_cast<uint8_t*>(&bars + 1);
  rest = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rest) + 15) & ~static_cast<uintptr_t>(15));
  ArrSelShared* selsh = reinterpret_cast<ArrSelShared*>(rest);
  uint32_t* keys = reinterpret_cast<uint32_t*>(selsh + 1);  // [kDecSegMax] keys in record order
  uint32_t* bkeys = keys + kDecSegMax;                      // block maxima of the segment (keys)
  // candidate mode: the record position where each 64-slot run of the segment starts
  int32_t* hstart = reinterpret_cast<int32_t*>(bkeys);
  // marked-candidate selection: one bit per entry of the segment
  uint32_t* listed = bkeys + p.seg_table;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = blockIdx.y, seg = blockIdx.x, n_seg = gridDim.x;
  const bool do_topk = p.K > 0;
  ArrSel<kThreads / 32> sel;  // the whole block, once the stream is done
  sel.sh = selsh;
  sel.tid = tid;
  const bool fast = do_topk && p.cluster_merge && p.fast_select;

  // ---- set-up that reads no input: it overlaps the previous kernel's tail (programmatic
  // dependent launch)
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc05::mbar_init(&bars.full[s], 1);
      tc05::mbar_init(&bars.empty[s], 1);
    }
    tc05::mbar_init(&bars.qready, kDecEpiWarps);  // FP8: the epilogue warps built the E4M3 terms
    for (int a = 0; a < 2; ++a) {
      tc05::mbar_init(&bars.tfull[a], 1);
      tc05::mbar_init(&bars.tempty[a], kDecEpiWarps / 2);  // one arrive per warp of the draining group
    }
    tc05::mbar_init(&bars.qfull, 1);
    bars.timeout = 0;
    bars.issued = bars.consumed = bars.drained = 0;
    for (int i = 0; i < 16; ++i) bars.tile_keys[i] = 0;
    bars.maxkey = 0u;
    bars.lister_fail = 0;
    tc05::fence_barrier_init();
  }
  if (warp == 1) tc05::tmem_alloc(&bars.tmem_base, C::kTmemCols);
  // the whole block-maxima table (this segment's blocks are known once the inputs are read)
  if (p.block_max)
    for (int i = tid; i < p.seg_table; i += kThreads) bkeys[i] = 0u;
  if (do_topk) sel.zero_hist(kHistBins);
  if (fast)
    for (int i = tid; i < kDecSegMax / 32; i += kThreads) listed[i] = 0u;

  // ---- wait for the previous kernel in the stream before reading any input
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  const int b = p.seq_of_row[row];
  // Candidate mode (Reindex over a block pool): the row's records are its candidate slots,
  // ascending positions in runs of cand_run consecutive records; every 64-slot half of a tile
  // is one contiguous run, loaded by its own 64-row TMA box.
  const bool cmode = p.cand != nullptr;
  const long long L_row = cmode ? (long long)p.n_cand[row] : min((long long)p.n_visible[row], p.N);
  const int U = p.unit;
  const long long n_units = (L_row + U - 1) / U;
  long long u0, u1;
  split_range(n_units, n_seg, seg, u0, u1);
  const long long e0 = u0 * U, e1 = min(u1 * U, L_row);
  const int n_tiles = e1 > e0 ? (int)((e1 - e0 + kTileKeys - 1) / kTileKeys) : 0;
  const int seg_len = (int)(e1 - e0);
  const int bs = p.block_max ? U : 1;
  const int seg_blocks = p.block_max ? (int)((e1 - e0 + bs - 1) / bs) : 0;
  if (cmode)
    for (int i = tid; i < (seg_len + 63) / 64; i += kThreads)
      hstart[i] = p.cand[(size_t)row * p.cand_stride + e0 + 64 * i];
  tc05::fence_before();
  __syncthreads();
  tc05::fence_after();
  // the histograms are zeroed: the other blocks' listers may read this one after this phase
  if (fast) cluster_arrive();
  const uint32_t tmem = bars.tmem_base;
  // Every block of a single-wave grid is resident: a dependent kernel (the attention) may be
  // scheduled onto the SMs left free; it waits for this grid before it reads the indices.
  if (p.pdl_trigger) asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0 && n_tiles > 0) {
      if (!FP8) {
        tc05::mbar_expect_tx(&bars.qfull, 2 * kDecQHalf);
        tc05::tma_load_2d(qs, &tmQ, 0, row * 32, &bars.qfull);
        tc05::tma_load_2d(qs + kDecQHalf, &tmQ, 64, row * 32, &bars.qfull);
      }
      const int y0 = (int)((long long)b * p.N + e0);
      for (int t = 0; t < n_tiles; ++t) {
        const int s = t % kStages;
        if (!tc05::mbar_wait(&bars.empty[s], ((t / kStages) & 1) ^ 1)) {
          report_timeout(&bars.timeout, p.dev_status);
          break;
        }
        uint8_t* dst = ring + s * C::kTileBytes;
        if (FP8) {
          // one 128-byte row per record; candidate mode: one 64-row box per run
          if (cmode) {
            const int halves = min(2, (seg_len - t * kTileKeys + 63) / 64);
            tc05::mbar_expect_tx(&bars.full[s], (uint32_t)halves * (C::kTileBytes / 2));
            for (int h = 0; h < halves; ++h)
              tc05::tma_load_2d(dst + h * (C::kTileBytes / 2), &tmK64, 0, (int)((long long)b * p.N + hstart[2 * t + h]),
                                &bars.full[s]);
          } else {
            tc05::mbar_expect_tx(&bars.full[s], C::kTileBytes);
            tc05::tma_load_2d(dst, &tmK, 0, y0 + t * kTileKeys, &bars.full[s]);
          }
        } else if (cmode) {
          // one or two 64-slot runs (rows 0..63 and 64..127 of the tile's swizzled halves)
          const int halves = min(2, (seg_len - t * kTileKeys + 63) / 64);
          tc05::mbar_expect_tx(&bars.full[s], (uint32_t)halves * (kKeyTile / 2));
          for (int h = 0; h < halves; ++h) {
            const int y = (int)((long long)b * p.N + hstart[2 * t + h]);
            tc05::tma_load_2d(dst + h * (kKeyHalf / 2), &tmK64, 0, y, &bars.full[s]);
            tc05::tma_load_2d(dst + kKeyHalf + h * (kKeyHalf / 2), &tmK64, 64, y, &bars.full[s]);
          }
        } else {
          tc05::mbar_expect_tx(&bars.full[s], kKeyTile);
          tc05::tma_load_2d(dst, &tmK, 0, y0 + t * kTileKeys, &bars.full[s]);
          tc05::tma_load_2d(dst + kKeyHalf, &tmK, 64, y0 + t * kTileKeys, &bars.full[s]);
        }
        bars.issued = t + 1;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t idesc = FP8 ? tc05::idesc_e4m3(128, C::kN) : tc05::idesc_bf16(128, C::kN);
      bool ok = tc05::mbar_wait(FP8 ? &bars.qready : &bars.qfull, 0);
      const uint64_t qd = tc05::sw128_desc(smem_u32(qs));
      const uint64_t ring_d = tc05::sw128_desc(smem_u32(ring));
      for (int t = 0; ok && t < n_tiles; ++t) {
        const int s = t % kStages, a = t & 1;
        if (!tc05::mbar_wait(&bars.full[s], (t / kStages) & 1) ||
            !tc05::mbar_wait(&bars.tempty[a], ((t >> 1) & 1) ^ 1)) {
          ok = false;
          break;
        }
        tc05::fence_after();
        const uint64_t ad = tc05::desc_adv(ring_d, s * C::kTileBytes);
        const uint32_t d_t = tmem + (uint32_t)a * C::kAccCols;
        if (FP8) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc05::mma_e4m3(d_t, tc05::desc_adv(ad, kk * 32), tc05::desc_adv(qd, kk * 32), idesc, kk > 0);
        } else {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kKeyHalf + (kk & 3) * 32;
            const uint32_t qoff = (kk >> 2) * kDecQHalf + (kk & 3) * 32;
            tc05::mma_bf16(d_t, tc05::desc_adv(ad, off), tc05::desc_adv(qd, qoff), idesc, kk > 0);
          }
        }
        tc05::mma_commit(&bars.empty[s]);
        tc05::mma_commit(&bars.tfull[a]);
        bars.consumed = t + 1;
      }
      if (!ok) report_timeout(&bars.timeout, p.dev_status);
    }
    __syncwarp();
  } else if (warp == 2 && fast) {
    // ---------------------------------------------------------------- candidate lister
    cluster_wait();  // every block of the cluster has zeroed its histogram
    uint32_t bound = 0u, mx = 0u;
    bool have = false, ok = true;
    const int x1 = max(1, n_tiles / 2), x2 = max(x1 + 1, (3 * n_tiles) / 4);
#pragma unroll 1
    for (int t = 0; t < n_tiles; ++t) {
      if (!wait_tile_keys(bars.tile_keys, t)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = t * kTileKeys + 32 * u + lane;
        if (j < seg_len) mx = max(mx, keys[j]);
      }
      if (t + 1 == x1 || t + 1 == x2) {
        uint32_t m = mx;
#pragma unroll
        for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) *reinterpret_cast<volatile uint32_t*>(&bars.maxkey) = m;
        __syncwarp();
        bound = max(bound, row_key_bound(selsh->hist, &bars.maxkey, (uint32_t)n_seg, p.K));
        if (!have) {
#pragma unroll 1
          for (int t2 = 0; t2 < t; ++t2) mark_tile(listed, keys, t2, seg_len, bound);
          have = true;
        }
      }
      if (have) mark_tile(listed, keys, t, seg_len, bound);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) {
      bars.maxkey = mx;  // every key of the segment (all tiles were read)
      bars.bound = bound;
    }
    if (!ok && lane == 0) {
      bars.lister_fail = 1;
      report_timeout(&bars.timeout, p.dev_status);
    }
    __syncwarp();
  } else if (warp >= kDecEpiFirst) {
    // ---------------------------------------------------------------- epilogue
    // group g = 0 drains the even tiles (accumulator 0), group 1 the odd ones (accumulator 1);
    // each record's score goes to the key array (in record order) and the level-1 histogram
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const int grp = (warp - kDecEpiFirst) >> 2;
    float w[32];
#pragma unroll
    for (int h = 0; h < 32; ++h) w[h] = __ldg(p.w + (size_t)row * kIdxHeads + h);
    bool dead = false;
    if (FP8 && n_tiles > 0) {
      fp8_q_terms(p.q_idx, row, tid - kDecEpiFirst * 32, qs, bars.qexp);
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // the MMA reads B through the async proxy
      __syncwarp();
      if (lane == 0) tc05::mbar_arrive(&bars.qready);
      // the heads of q^I were scaled by 2^qexp[h]: the weights take the inverse factor
      dead = !tc05::mbar_wait(&bars.qready, 0);
      if (dead && lane == 0) report_timeout(&bars.timeout, p.dev_status);
#pragma unroll
      for (int h = 0; h < 32; ++h) w[h] *= __int_as_float((127 - bars.qexp[h]) << 23);
    }
    float* srow = p.scores ? p.scores + (size_t)row * p.scores_stride : nullptr;
    const float* kscale = FP8 ? p.k_scale + (size_t)b * p.N : nullptr;
    const int n_pairs = (n_tiles + 1) / 2;
    // FP8: the scale of this thread's record in the group's next tiles, loaded kScalePre
    // tiles ahead (an HBM load per tile would otherwise stall every iteration)
    constexpr int kScalePre = 4;
    auto scale_of = [&](int pr) -> float {
      const int jl = (2 * pr + grp) * kTileKeys + 32 * quarter + lane;
      return jl < seg_len ? __ldg(kscale + (cmode ? hstart[jl >> 6] + (jl & 63) : e0 + jl)) : 1.f;
    };
    float kpre[kScalePre];
#pragma unroll
    for (int i = 0; i < kScalePre; ++i) kpre[i] = FP8 ? scale_of(i) : 1.f;
    for (int pr = 0; pr < n_pairs; ++pr) {
      const int t = 2 * pr + grp, a = grp;
      if (t >= n_tiles) continue;
      if (!dead && !tc05::mbar_wait(&bars.tfull[a], pr & 1)) {
        dead = true;
        if (lane == 0) report_timeout(&bars.timeout, p.dev_status);
      }
      float sc = 0.f;
      const int jl = t * kTileKeys + 32 * quarter + lane;  // record index within the segment
      const float ksc = kpre[0];
      if (FP8) {
#pragma unroll
        for (int i = 0; i + 1 < kScalePre; ++i) kpre[i] = kpre[i + 1];
        kpre[kScalePre - 1] = scale_of(pr + kScalePre);
      }
      if (!dead) {
        tc05::fence_after();
        const uint32_t d_t = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)a * C::kAccCols;
        uint32_t v[32];
        tc05::tmem_ld32(d_t, v);
        if (FP8) {
          // D1 + (D2 + D3 / 16) / 16 per head
          uint32_t v2[32], v3[32];
          tc05::tmem_ld32(d_t + 32, v2);
          tc05::tmem_ld32(d_t + 64, v3);
          tc05::tmem_ld_wait();
          tc05::fence_before();
          __syncwarp();
          if (lane == 0) tc05::mbar_arrive(&bars.tempty[a]);
#pragma unroll
          for (int h = 0; h < 32; ++h) {
            const float x = fmaf(fmaf(__uint_as_float(v3[h]), 0.0625f, __uint_as_float(v2[h])), 0.0625f,
                                 __uint_as_float(v[h]));
            sc = fmaf(w[h], fmaxf(x * ksc, 0.f), sc);
          }
        } else {
          tc05::tmem_ld_wait();
          tc05::fence_before();
          __syncwarp();
          if (lane == 0) tc05::mbar_arrive(&bars.tempty[a]);
#pragma unroll
          for (int h = 0; h < 32; ++h) sc = fmaf(w[h], fmaxf(__uint_as_float(v[h]), 0.f), sc);
        }
        if (warp == kDecEpiFirst + 4 * grp && lane == 0) atomicMax(&bars.drained, t + 1);
      }
      const bool valid = !dead && jl < seg_len;
      const uint32_t key = valid ? score_key(sc) : 0u;
      if (do_topk && jl < seg_len) {
        keys[jl] = key;
        if (valid) atomicAdd(&selsh->hist[key >> 20], 1);
      }
      if (fast) {  // this warp's keys of tile t are stored: one count for the lister
        __syncwarp();
        if (lane == 0) {
          __threadfence_block();
          atomicAdd(&bars.tile_keys[t & 15], 1);
        }
      }
      if (srow && valid) srow[e0 + jl] = sc;
      if (seg_blocks) {
        // block maxima: a warp's 32 records lie in one block when bs >= 32 (one atomic per warp)
        if (bs >= 32) {
          const uint32_t m = __reduce_max_sync(0xffffffffu, key);
          if (lane == 0 && m != 0u) atomicMax(&bkeys[(t * kTileKeys + 32 * quarter) / bs], m);
        } else if (valid) {
          atomicMax(&bkeys[jl / bs], key);
        }
      }
    }
  }

  // ---------------------------------------------------------------- tail (whole block)
  __syncthreads();
  {
    // Once every tile has been drained no copy or MMA touches the ring and the query tile any
    // more (the copies and MMAs completed through the mbarriers the epilogue waited on), so
    // they serve as the selection's scratch: the candidate lists, and the selected entries'
    // indices (CSA2_MAX_TOPK words at the end).  After a timeout copies may be in flight: the
    // selection is skipped (the status reports the timeout).
    constexpr int kScratchWords = (kDecRingBytes + C::kQBytes) / 4;
    constexpr int kListRoom = kScratchWords - CSA2_MAX_TOPK;
    static_assert(ArrSel<kThreads / 32>::list_words(kDecSegMax) <= kListRoom, "selection lists fit in the scratch");
    static_assert(2 * kFastCap + ArrSel<kThreads / 32>::list_words(kFastCap) <= kListRoom,
                  "marked entries and their selection lists fit in the scratch");
    sel.scratch = reinterpret_cast<uint32_t*>(ring);
    int32_t* sel_idx = reinterpret_cast<int32_t*>(ring) + kListRoom;
    // record position of the segment's entry i
    auto pos_of = [&](int i) -> int32_t { return cmode ? hstart[i >> 6] + (i & 63) : (int32_t)(e0 + i); };
    const bool live = !bars.timeout;
    for (int i = tid; i < seg_blocks; i += kThreads)
      p.block_max[(size_t)row * p.bmax_stride + e0 / bs + i] = bkeys[i] ? key_score(bkeys[i]) : -INFINITY;
    if (seg == n_seg - 1) {
      float* srow = p.scores ? p.scores + (size_t)row * p.scores_stride : nullptr;
      if (srow)
        for (long long jj = L_row + tid; jj < p.scores_len; jj += kThreads) srow[jj] = -INFINITY;
      if (p.block_max)
        for (long long blk = (L_row + bs - 1) / bs + tid; blk < p.n_blocks; blk += kThreads)
          p.block_max[(size_t)row * p.bmax_stride + blk] = -INFINITY;
    }
    bool fast_done = false;
    if (fast) {
      // ------------------------------------------------ selection among the marked entries
      const uint32_t rank = cluster_rank();
      if (warp != 2) cluster_wait();  // (the lister warp waited for this phase already)
      // this block's marked entries, in entry order: keys at ring[0 ..), record positions at
      // ring[kFastCap ..)
      uint32_t* ck = reinterpret_cast<uint32_t*>(ring);
      int32_t* cp = reinterpret_cast<int32_t*>(ring) + kFastCap;
      const int n_words = (seg_len + 31) / 32;
      uint32_t wa = 0u, wb = 0u;  // thread t: bitmap words 2t, 2t + 1
      if (live && 2 * tid < n_words) wa = listed[2 * tid];
      if (live && 2 * tid + 1 < n_words) wb = listed[2 * tid + 1];
      int n_mine;
      int at = sel.scan(__popc(wa) + __popc(wb), &n_mine);
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        uint32_t m = h ? wb : wa;
        const int base = 32 * (2 * tid + h);
        while (m) {
          const int i = base + __ffs(m) - 1;
          m &= m - 1u;
          if (at < kFastCap) {
            ck[at] = keys[i];
            cp[at] = pos_of(i);
          }
          ++at;
        }
      }
      // every block learns every block's count (pushed into each block's table)
      if (tid < n_seg) {
        cluster_st_s32(cluster_map(&bars.cand_cnt[rank], (uint32_t)tid), (!live || bars.lister_fail) ? -1 : n_mine);
        cluster_st_s32(cluster_map(&bars.cand_lo[rank], (uint32_t)tid), (int)bars.bound);
        cluster_st_s32(cluster_map(&bars.cand_hi[rank], (uint32_t)tid), (int)bars.maxkey);
      }
      cluster_sync();  // every block's marked entries and count are published
      if (warp == 0) {
        const int c = lane < n_seg ? bars.cand_cnt[lane] : 0;
        const bool bad = __any_sync(0xffffffffu, c < 0);
        int inc = max(c, 0);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += y;
        }
        if (lane <= n_seg) bars.cand_off[lane] = inc - max(c, 0);
        const int total = __shfl_sync(0xffffffffu, inc, 31);
        if (lane == 0) bars.cand_go = !bad && total <= kFastCap;
      }
      __syncthreads();
      if (bars.cand_go) {
        fast_done = true;
        const int total = bars.cand_off[n_seg];
        if (rank == 0) {
          // the selection's histograms start at zero
          for (int i = tid; i < kHistBins; i += kThreads) selsh->hist[i] = 0;
          if (tid < 128) selsh->aux[tid] = 0u;
          // block 0 appends the other blocks' lists to its own (same layout in every block)
          // (16-byte loads of four entries; a list's last group may read up to three words past
          // its end, inside the ring)
#pragma unroll 1
          for (int g = tid;; g += kThreads) {
            int r = 1, g0 = 0;
            while (r < n_seg && g >= g0 + (bars.cand_off[r + 1] - bars.cand_off[r] + 3) / 4) {
              g0 += (bars.cand_off[r + 1] - bars.cand_off[r] + 3) / 4;
              ++r;
            }
            if (r >= n_seg) break;
            const int i = 4 * (g - g0), n_r = bars.cand_off[r + 1] - bars.cand_off[r], f = bars.cand_off[r] + i;
            const uint4 kv = cluster_ld_v4(cluster_map(ck + i, (uint32_t)r));
            const uint4 pv = cluster_ld_v4(cluster_map(cp + i, (uint32_t)r));
            const uint32_t kk[4] = {kv.x, kv.y, kv.z, kv.w}, pp[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (i + u < n_r) {
                ck[f + u] = kk[u];
                cp[f + u] = (int32_t)pp[u];
              }
          }
          __syncthreads();
          cluster_arrive();  // the other blocks' shared memory is no longer read
          uint32_t lo = 0u, hi = 0u;
          for (int r = 0; r < n_seg; ++r) {
            lo = max(lo, bars.cand_lo[r]);
            hi = max(hi, bars.cand_hi[r]);
          }
          select_marked(sel, ck, cp, total, p.K, lo, hi, p.idx + (size_t)row * p.K);
          cluster_wait();
        } else {
          cluster_arrive();
          cluster_wait();
        }
      }
    }
    if (fast_done) {
      // (block 0 wrote the row's indices)
    } else if (do_topk && p.cluster_merge) {
      // The row's segments form a thread-block cluster (rank = segment): the histogram
      // levels are summed over the cluster, so the blocks select the row's top-K together and
      // each writes its share of the row's indices at its offset; no lists leave the chip.
      // Every block takes part in every cluster step, also after a timeout (then with no
      // entries: the status reports the timeout).
      const uint32_t rank = cluster_rank();
      const int n_here = live ? seg_len : 0;
      arr_threshold_impl(sel, keys, n_here, p.K, true, ClusterPick<kThreads / 32>{rank, (uint32_t)n_seg, kDecSegMax});
      int base = 0, total = 0, kept = 0;
      if (selsh->thr == 0u) {
        // at most K candidates in the row: every block keeps all its entries; offsets by
        // exchanging the blocks' counts
        kept = arr_compact_cluster(sel, n_here, sel_idx, rank, (uint32_t)n_seg, &base, &total);
      } else {
        // block 0 wrote this block's number of ties to keep, its offset and the row's total
        base = (int)selsh->aux[2];
        total = (int)selsh->aux[4];
        kept = arr_compact(sel, n_here, sel_idx);
      }
      int32_t* out = p.idx + (size_t)row * p.K;
      for (int r = tid; r < kept; r += kThreads)
        if (base + r < p.K) out[base + r] = pos_of(sel_idx[r]);
      if (rank == (uint32_t)n_seg - 1)
        for (int r = total + tid; r < p.K; r += kThreads) out[r] = -1;
      // (the selection's last cluster barrier follows every access to another block's
      // shared memory, so the blocks may leave independently)
    } else if (do_topk && live) {
      arr_threshold(sel, keys, seg_len, p.K, true);
      const int kept = arr_compact(sel, seg_len, sel_idx);
      if (n_seg == 1) {
        int32_t* out = p.idx + (size_t)row * p.K;
        for (int r = tid; r < p.K; r += kThreads) out[r] = r < kept ? pos_of(sel_idx[r]) : -1;
      } else {
        const size_t o = ((size_t)row * n_seg + seg) * p.K;
        for (int r = tid; r < kept; r += kThreads) {
          p.seg_keys[o + r] = keys[sel_idx[r]];
          p.seg_pos[o + r] = pos_of(sel_idx[r]);
        }
        if (tid == 0) {
          p.seg_cnt[(size_t)row * n_seg + seg] = kept;
          p.seg_thr[(size_t)row * n_seg + seg] = kept >= p.K ? selsh->thr : 0u;
        }
        if (p.row_done != nullptr) {
          // The last segment of the row to finish merges every segment's list (no waiting:
          // the block that sees the count reach n_seg - 1 knows the others have published).
          // The counter carries the call's tag in its high half: a stale value from an
          // earlier call restarts at 1, so the workspace needs no clearing between calls.
          __threadfence();
          __syncthreads();
          if (tid == 0) bars.last = count_arrival(p.row_done + row, p.call_tag, n_seg, p.dev_status);
          __syncthreads();
          if (bars.last) {
            __threadfence();
            merge_row_lists(sel, keys, p, row, n_seg, sel_idx, kListRoom);
          }
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (bars.timeout && tid == 0) {
    // drain loads and MMAs still in flight (bounded), then free tensor memory
    // (only the last kStages loads can be outstanding: each stage's latest phase)
    for (int t = max(0, bars.issued - kStages); t < bars.issued; ++t)
      tc05::mbar_wait(&bars.full[t % kStages], (t / kStages) & 1);
    for (int t = max(0, bars.drained - 1); t < bars.consumed; ++t)
      tc05::mbar_wait(&bars.tfull[t & 1], (t >> 1) & 1);
  }
  __syncthreads();
  if (warp == 1) {
    tc05::fence_after();
    tc05::tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ============================================================================ FP8 decode, streaming
// FP8 decode rows too long for one wave of the decode kernel's segments (every key of a
// segment stays in that kernel's shared memory): the same tile pipeline (TMA ring, four
// kind::f8f6f4 MMAs per 128-record tile against the E4M3 terms of q^I, two accumulators in
// tensor memory, two groups of four epilogue warps on alternate tiles), but the epilogue feeds
// the exact streaming top-K engine (select.cuh: per-warp buffers of about K entries, entries
// below the running K-th key dropped on arrival) instead of keeping every key.  A block then
// needs about 110 KB of shared memory and 256 tensor-memory columns, so two blocks share an
// SM: one block streams FP8 tiles at about two thirds of an SM's share of the HBM rate (its
// copy thread, MMA thread and epilogue warps form one dependent chain per tile and contend
// for the SM's issue slots), two blocks per SM interleave two such chains.
// The epilogue checks the buffers every 4 tiles; one near capacity is first pruned by one
// histogram pass (eng_prune), the exact select runs only when that leaves too little room,
// since the stream waits on the epilogue meanwhile.  At the end the exact select leaves the
// segment's K best, placed in position order through a bitmap of their offsets in the idle
// ring (or, for a segment longer than the bitmap, by the engine's searches).  Each block
// writes its segment's list (at most K entries in position order, and its K-th key) for the
// lists merge, or the row's indices when the row is a single segment.
constexpr int kStrStages = 3;
constexpr int kStrTile = kTileKeys * 128;  // 16 KB: 128 records x 128 E4M3 dims
constexpr int kStrThreads = 12 * 32;       // warp 0 TMA, warp 1 MMA + tensor memory, warps 4..11 epilogue
constexpr int kStrEpiFirst = 4;
constexpr int kStrEpiWarps = 8;
constexpr int kStrQBytes = 96 * 128;       // B: the three E4M3 terms of the 32 heads
constexpr uint32_t kStrAccCols = 128;      // columns per accumulator (96 used)
constexpr uint32_t kStrTmemCols = 256;
constexpr int kStrRound = kRoundEntries / 32;  // tiles per epilogue warp between engine checks

struct StrBars {
  alignas(16) float w[32];  // head weights times the inverse of q^I's head scale
  uint64_t full[kStrStages], empty[kStrStages], tfull[2], tempty[2], qready;
  uint32_t tmem_base;
  int timeout;
  int issued;    // tiles whose TMA loads were issued
  int consumed;  // tiles whose MMAs were issued
  int drained;   // tiles whose accumulators the epilogue read
  int bitmap;    // the survivors are placed through a position bitmap in the idle ring
  int qexp[32];  // power-of-two exponent applied to each head of q^I
};

__host__ __device__ constexpr size_t str_align16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

size_t str_smem_bytes(int K) {
  return 1024 + (size_t)kStrStages * kStrTile + kStrQBytes + str_align16(sizeof(StrBars)) +
         str_align16(sizeof(EngShared)) + (size_t)kStrEpiWarps * (K + kRoundEntries) * 8 + (size_t)K * 8;
}

__global__ void __launch_bounds__(kStrThreads, 2)
    idx_fp8_stream_kernel(const __grid_constant__ CUtensorMap tmK, const ScanParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* ring = smem;
  uint8_t* qs = ring + kStrStages * kStrTile;
  StrBars& bars = *reinterpret_cast<StrBars*>(qs + kStrQBytes);
  uint8_t* rest = reinterpret_cast<uint8_t*>(&bars) + str_align16(sizeof(StrBars));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = blockIdx.y, seg = blockIdx.x, n_seg = gridDim.x;
  Engine<kStrEpiWarps> eng;  // the epilogue warps (named barrier 1)
  eng.sh = reinterpret_cast<EngShared*>(rest);
  eng.cap = p.K + kRoundEntries;
  eng.keys = reinterpret_cast<uint32_t*>(rest + str_align16(sizeof(EngShared)));
  eng.js = reinterpret_cast<int32_t*>(eng.keys + kStrEpiWarps * eng.cap);
  eng.out_key = reinterpret_cast<uint32_t*>(eng.js + kStrEpiWarps * eng.cap);
  eng.out_j = reinterpret_cast<int32_t*>(eng.out_key + p.K);
  eng.bar_id = 1;
  eng.tid = tid - kStrEpiFirst * 32;

  // ---- set-up that reads no input (overlaps the previous kernel's tail)
  if (tid == 0) {
    for (int s = 0; s < kStrStages; ++s) {
      tc05::mbar_init(&bars.full[s], 1);
      tc05::mbar_init(&bars.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc05::mbar_init(&bars.tfull[a], 1);
      tc05::mbar_init(&bars.tempty[a], 4);  // one arrive per warp of the draining group
    }
    tc05::mbar_init(&bars.qready, kStrEpiWarps);
    bars.timeout = 0;
    bars.issued = bars.consumed = bars.drained = 0;
    tc05::fence_barrier_init();
  }
  if (warp == 1) tc05::tmem_alloc(&bars.tmem_base, kStrTmemCols);

  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  const int b = p.seq_of_row[row];
  const long long L_row = max(0LL, min((long long)p.n_visible[row], p.N));
  long long u0, u1;
  split_range((L_row + kTileKeys - 1) / kTileKeys, n_seg, seg, u0, u1);
  const long long e0 = u0 * kTileKeys, e1 = min(u1 * kTileKeys, L_row);
  const int n_tiles = e1 > e0 ? (int)((e1 - e0 + kTileKeys - 1) / kTileKeys) : 0;
  const int seg_len = e1 > e0 ? (int)(e1 - e0) : 0;
  tc05::fence_before();
  __syncthreads();
  tc05::fence_after();
  const uint32_t tmem = bars.tmem_base;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0 && n_tiles > 0) {
      const long long y0 = (long long)b * p.N + e0;
      for (int t = 0; t < n_tiles; ++t) {
        const int s = t % kStrStages;
        if (!tc05::mbar_wait(&bars.empty[s], ((t / kStrStages) & 1) ^ 1)) {
          report_timeout(&bars.timeout, p.dev_status);
          break;
        }
        tc05::mbar_expect_tx(&bars.full[s], kStrTile);
        tc05::tma_load_2d(ring + s * kStrTile, &tmK, 0, (int)(y0 + (long long)t * kTileKeys), &bars.full[s]);
        bars.issued = t + 1;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t idesc = tc05::idesc_e4m3(128, 96);
      bool ok = tc05::mbar_wait(&bars.qready, 0);
      const uint64_t qd = tc05::sw128_desc(smem_u32(qs));
      const uint64_t ring_d = tc05::sw128_desc(smem_u32(ring));
      for (int t = 0; ok && t < n_tiles; ++t) {
        const int s = t % kStrStages, a = t & 1;
        if (!tc05::mbar_wait(&bars.full[s], (t / kStrStages) & 1) ||
            !tc05::mbar_wait(&bars.tempty[a], ((t >> 1) & 1) ^ 1)) {
          ok = false;
          break;
        }
        tc05::fence_after();
        const uint64_t ad = tc05::desc_adv(ring_d, s * kStrTile);
        const uint32_t d_t = tmem + (uint32_t)a * kStrAccCols;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc05::mma_e4m3(d_t, tc05::desc_adv(ad, kk * 32), tc05::desc_adv(qd, kk * 32), idesc, kk > 0);
        tc05::mma_commit(&bars.empty[s]);
        tc05::mma_commit(&bars.tfull[a]);
        bars.consumed = t + 1;
      }
      if (!ok) report_timeout(&bars.timeout, p.dev_status);
    }
    __syncwarp();
  } else if (warp >= kStrEpiFirst) {
    // ---------------------------------------------------------------- epilogue + top-K
    // group 0 drains the even tiles (accumulator 0), group 1 the odd ones; each warp's
    // records arrive in ascending position order, as the engine's buffers require
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const int grp = (warp - kStrEpiFirst) >> 2;
    eng_init(eng);
    bool dead = false;
    if (n_tiles > 0) {
      fp8_q_terms(p.q_idx, row, eng.tid, qs, bars.qexp);
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // the MMA reads B through the async proxy
      __syncwarp();
      if (lane == 0) tc05::mbar_arrive(&bars.qready);
      dead = !tc05::mbar_wait(&bars.qready, 0);
      if (dead && lane == 0) report_timeout(&bars.timeout, p.dev_status);
      // the heads of q^I were scaled by 2^qexp[h]: the weights take the inverse factor (kept
      // in shared memory, read as broadcasts: registers are scarce at two blocks per SM)
      if (eng.tid < 32)
        bars.w[eng.tid] = __ldg(p.w + (size_t)row * kIdxHeads + eng.tid) * __int_as_float((127 - bars.qexp[eng.tid]) << 23);
      eng.sync();
    }
    const float4* w4 = reinterpret_cast<const float4*>(bars.w);
    const float* kscale = p.k_scale + (size_t)b * p.N + e0;
    // the scale of this thread's record in the group's next tiles, loaded kScalePre tiles ahead
    constexpr int kScalePre = 4;
    auto scale_of = [&](int pr) -> float {
      const int jl = (2 * pr + grp) * kTileKeys + 32 * quarter + lane;
      return jl < seg_len ? __ldg(kscale + jl) : 1.f;
    };
    float kpre[kScalePre];
#pragma unroll
    for (int i = 0; i < kScalePre; ++i) kpre[i] = scale_of(i);
    const int n_pairs = (n_tiles + 1) / 2;
    int cnt = 0;
    uint32_t thr = 0u;
    for (int pr = 0; pr < n_pairs; ++pr) {
      const int t = 2 * pr + grp, a = grp;
      const bool have = t < n_tiles;
      const int jl = t * kTileKeys + 32 * quarter + lane;  // record index within the segment
      const float ksc = kpre[0];
#pragma unroll
      for (int i = 0; i + 1 < kScalePre; ++i) kpre[i] = kpre[i + 1];
      kpre[kScalePre - 1] = scale_of(pr + kScalePre);
      if (have && !dead && !tc05::mbar_wait(&bars.tfull[a], pr & 1)) {
        dead = true;
        if (lane == 0) report_timeout(&bars.timeout, p.dev_status);
      }
      float sc = 0.f;
      if (have && !dead) {
        tc05::fence_after();
        const uint32_t d_t = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)a * kStrAccCols;
        // D1 + (D2 + D3 / 16) / 16 per head, eight heads at a time
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          uint32_t v1[8], v2[8], v3[8];
          tc05::tmem_ld8(d_t + 8 * c8, v1);
          tc05::tmem_ld8(d_t + 32 + 8 * c8, v2);
          tc05::tmem_ld8(d_t + 64 + 8 * c8, v3);
          tc05::tmem_ld_wait();
          const float4 wa = w4[2 * c8], wb = w4[2 * c8 + 1];
          const float wc[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float x = fmaf(fmaf(__uint_as_float(v3[i]), 0.0625f, __uint_as_float(v2[i])), 0.0625f,
                                 __uint_as_float(v1[i]));
            sc = fmaf(wc[i], fmaxf(x * ksc, 0.f), sc);
          }
        }
        tc05::fence_before();
        __syncwarp();
        if (lane == 0) tc05::mbar_arrive(&bars.tempty[a]);
        if (warp == kStrEpiFirst + 4 * grp && lane == 0) atomicMax(&bars.drained, t + 1);
      }
      const bool valid = have && !dead && jl < seg_len;
      eng_append(eng, cnt, thr, valid, score_key(sc), (int32_t)(e0 + jl));
      // (a buffer near capacity: one-pass prune, the exact select only when that leaves too
      // little room; the stream waits on the epilogue meanwhile)
      if (pr % kStrRound == kStrRound - 1 || pr == n_pairs - 1) thr = eng_check_fast(eng, p.K, cnt);
    }
    // ---- the segment's K best, in position order
    constexpr int NT = kStrEpiWarps * 32;
    if (lane == 0) eng.sh->warp_cnt[eng.warp()] = cnt;
    eng.sync();
    eng_select(eng, p.K);
    uint32_t* thr_out = n_seg > 1 ? p.seg_thr + (size_t)row * n_seg + seg : nullptr;
    // Survivors' ranks through a bitmap of their positions in the segment and a prefix over
    // its words (the ring is idle once every tile was drained; after a timeout copies may
    // still land there, and segments longer than the bitmap rank by binary search instead).
    constexpr int kBitmapWords = kStrStages * kStrTile / 8;  // bitmap, then its word prefixes
    const int nw = (seg_len + 31) / 32;
    if (eng.tid == 0) bars.bitmap = !bars.timeout && nw <= kBitmapWords;
    eng.sync();
    int n;
    if (bars.bitmap) {
      uint32_t* bm = reinterpret_cast<uint32_t*>(ring);
      int32_t* pre = reinterpret_cast<int32_t*>(bm + nw);
      const int w = eng.warp(), mycnt = eng.sh->warp_cnt[w];
      const uint32_t* gk = eng.keys + w * eng.cap;
      const int32_t* gj = eng.js + w * eng.cap;
      for (int i = eng.tid; i < nw; i += NT) bm[i] = 0u;
      eng.sync();
      for (int i = lane; i < mycnt; i += 32) {
        const int off = (int)(gj[i] - e0);
        atomicOr(&bm[off >> 5], 1u << (off & 31));
      }
      eng.sync();
      const int per = (nw + NT - 1) / NT, w0 = min(nw, eng.tid * per), w1 = min(nw, w0 + per);
      int local = 0;
      for (int i = w0; i < w1; ++i) local += __popc(bm[i]);
      int total_bits;
      int before = eng.scan(local, &total_bits);
      for (int i = w0; i < w1; ++i) {
        pre[i] = before;
        before += __popc(bm[i]);
      }
      eng.sync();
      for (int i = lane; i < mycnt; i += 32) {
        const int off = (int)(gj[i] - e0);
        const int r = pre[off >> 5] + __popc(bm[off >> 5] & ((1u << (off & 31)) - 1u));
        eng.out_key[r] = gk[i];
        eng.out_j[r] = gj[i];
      }
      n = total_bits;
      if (eng.tid == 0 && thr_out) *thr_out = n >= p.K ? eng.sh->thr : 0u;
      eng.sync();
    } else {
      n = eng_rank(eng, p.K, thr_out);
    }
    if (n_seg == 1) {
      int32_t* out = p.idx + (size_t)row * p.K;
      for (int i = eng.tid; i < p.K; i += NT) out[i] = i < n ? eng.out_j[i] : -1;
    } else {
      const size_t o = ((size_t)row * n_seg + seg) * p.K;
      for (int i = eng.tid; i < n; i += NT) {
        p.seg_keys[o + i] = eng.out_key[i];
        p.seg_pos[o + i] = eng.out_j[i];
      }
      if (eng.tid == 0) p.seg_cnt[(size_t)row * n_seg + seg] = n;
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (bars.timeout && tid == 0) {
    // drain loads and MMAs still in flight (bounded), then free tensor memory
    for (int t = max(0, bars.issued - kStrStages); t < bars.issued; ++t)
      tc05::mbar_wait(&bars.full[t % kStrStages], (t / kStrStages) & 1);
    for (int t = max(0, bars.drained - 1); t < bars.consumed; ++t)
      tc05::mbar_wait(&bars.tfull[t & 1], (t >> 1) & 1);
  }
  __syncthreads();
  if (warp == 1) {
    tc05::fence_after();
    tc05::tmem_dealloc(tmem, kStrTmemCols);
  }
}

// ===================================================================================== prefill
constexpr int kPreNQ = 8;                         // queries per MMA tile (N = 256)
constexpr int kPreN = 32 * kPreNQ;
constexpr int kPreStages = 4;
constexpr int kPreEpiFirst = 4;
constexpr int kPreEpiWarps = 8;
constexpr int kPreThreads = (kPreEpiFirst + kPreEpiWarps) * 32;  // 384
constexpr int kPreQHalf = kPreN * 128;            // 32 KB
constexpr uint32_t kPreTmemCols = 2 * kPreN;      // 512: two accumulators

struct PreBars {
  uint64_t full[kPreStages], empty[kPreStages], tfull[2], tempty[2], qfull, qempty;
  uint32_t tmem_base;
  int timeout;
  int issued, consumed, drained, q_issued, q_used;
  float w[kPreNQ][32];
  int nv[kPreNQ];
};

struct PreItem {
  int qt;        // query tile
  int t0, t1;    // key tiles [t0, t1)
};

// Work item i of the grid: query tile i / n_parts and the part-th share of its key tiles.
__device__ __forceinline__ PreItem pre_item(const ScanParams& p, int i, int n_parts) {
  PreItem it;
  it.qt = i / n_parts;
  const int part = i % n_parts;
  // the tile's key range is the widest causal range among its rows
  long long L = 0;
  for (int r = it.qt * kPreNQ; r < min(p.n_rows, (it.qt + 1) * kPreNQ); ++r)
    L = max(L, min((long long)p.n_visible[r], p.N));
  const int nt = (int)((L + kTileKeys - 1) / kTileKeys);
  it.t0 = (int)(((long long)nt * part) / n_parts);
  it.t1 = (int)(((long long)nt * (part + 1)) / n_parts);
  return it;
}

__global__ void __launch_bounds__(kPreThreads, 1)
    idx_mma_prefill_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                           const ScanParams p, int n_items, int n_parts) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* ring = smem;
  uint8_t* qs = ring + kPreStages * kKeyTile;
  PreBars& bars = *reinterpret_cast<PreBars*>(qs + 2 * kPreQHalf);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kPreStages; ++s) {
      tc05::mbar_init(&bars.full[s], 1);
      tc05::mbar_init(&bars.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc05::mbar_init(&bars.tfull[a], 1);
      tc05::mbar_init(&bars.tempty[a], kPreEpiWarps);
    }
    tc05::mbar_init(&bars.qfull, 1);
    tc05::mbar_init(&bars.qempty, 1);
    bars.timeout = 0;
    bars.issued = bars.consumed = bars.drained = bars.q_issued = bars.q_used = 0;
    tc05::fence_barrier_init();
  }
  if (warp == 1) tc05::tmem_alloc(&bars.tmem_base, kPreTmemCols);
  tc05::fence_before();
  __syncthreads();
  tc05::fence_after();
  const uint32_t tmem = bars.tmem_base;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int t_glob = 0, n_item = 0;  // n_item counts the non-empty items (Q-buffer phases)
      bool ok = true;
      for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x) {
        const PreItem it = pre_item(p, i, n_parts);
        if (it.t1 <= it.t0) continue;
        // the query tile buffer is free once every MMA of the previous item has completed
        if (!tc05::mbar_wait(&bars.qempty, (n_item & 1) ^ 1)) {
          ok = false;
          break;
        }
        tc05::mbar_expect_tx(&bars.qfull, 2 * kPreQHalf);
        tc05::tma_load_2d(qs, &tmQ, 0, it.qt * kPreN, &bars.qfull);
        tc05::tma_load_2d(qs + kPreQHalf, &tmQ, 64, it.qt * kPreN, &bars.qfull);
        bars.q_issued = n_item + 1;
        for (int t = it.t0; t < it.t1; ++t, ++t_glob) {
          const int s = t_glob % kPreStages;
          if (!tc05::mbar_wait(&bars.empty[s], ((t_glob / kPreStages) & 1) ^ 1)) {
            ok = false;
            break;
          }
          tc05::mbar_expect_tx(&bars.full[s], kKeyTile);
          uint8_t* dst = ring + s * kKeyTile;
          tc05::tma_load_2d(dst, &tmK, 0, t * kTileKeys, &bars.full[s]);
          tc05::tma_load_2d(dst + kKeyHalf, &tmK, 64, t * kTileKeys, &bars.full[s]);
          bars.issued = t_glob + 1;
        }
        ++n_item;
      }
      if (!ok) report_timeout(&bars.timeout, p.dev_status);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc05::idesc_bf16(128, kPreN);
      const uint32_t q_u = smem_u32(qs);
      int t_glob = 0, n_item = 0;  // non-empty items, as counted by the producer
      bool ok = true;
      for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x) {
        const PreItem it = pre_item(p, i, n_parts);
        if (it.t1 <= it.t0) continue;
        if (!tc05::mbar_wait(&bars.qfull, n_item & 1)) {
          ok = false;
          break;
        }
        for (int t = it.t0; t < it.t1; ++t, ++t_glob) {
          const int s = t_glob % kPreStages, a = t_glob & 1;
          if (!tc05::mbar_wait(&bars.full[s], (t_glob / kPreStages) & 1) ||
              !tc05::mbar_wait(&bars.tempty[a], ((t_glob >> 1) & 1) ^ 1)) {
            ok = false;
            break;
          }
          tc05::fence_after();
          const uint32_t a_u = smem_u32(ring + s * kKeyTile);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kKeyHalf + (kk & 3) * 32;
            const uint32_t qoff = (kk >> 2) * kPreQHalf + (kk & 3) * 32;
            tc05::mma_bf16(tmem + a * kPreN, tc05::sw128_desc(a_u + off), tc05::sw128_desc(q_u + qoff), idesc,
                           kk > 0);
          }
          tc05::mma_commit(&bars.empty[s]);
          tc05::mma_commit(&bars.tfull[a]);
          bars.consumed = t_glob + 1;
        }
        if (ok) {
          tc05::mma_commit(&bars.qempty);
          bars.q_used = n_item + 1;
        }
        ++n_item;
      }
      if (!ok) report_timeout(&bars.timeout, p.dev_status);
    }
    __syncwarp();
  } else if (warp >= kPreEpiFirst) {
    // ---------------------------------------------------------------- epilogue
    const int e = warp - kPreEpiFirst;       // 0..7
    const int quarter = warp & 3;            // TMEM lanes 32*quarter .. +31
    const int qhalf = e >> 2;                // queries 4*qhalf .. +3
    const int etid = tid - kPreEpiFirst * 32;
    int t_glob = 0;
    bool dead = false;
    for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
      const PreItem it = pre_item(p, i, n_parts);
      if (it.t1 <= it.t0) continue;
      asm volatile("bar.sync 1, %0;\n" ::"n"(kPreEpiWarps * 32) : "memory");
      if (etid < kPreNQ * 32) {
        const int c = etid >> 5, h = etid & 31, r = it.qt * kPreNQ + c;
        bars.w[c][h] = r < p.n_rows ? __ldg(p.w + (size_t)r * kIdxHeads + h) : 0.f;
        if (h == 0) bars.nv[c] = r < p.n_rows ? (int)min((long long)p.n_visible[r], p.N) : 0;
      }
      asm volatile("bar.sync 1, %0;\n" ::"n"(kPreEpiWarps * 32) : "memory");
      for (int t = it.t0; t < it.t1; ++t, ++t_glob) {
        const int a = t_glob & 1;
        if (!dead && !tc05::mbar_wait(&bars.tfull[a], (t_glob >> 1) & 1)) {
          dead = true;
          if (lane == 0) report_timeout(&bars.timeout, p.dev_status);
        }
        if (dead) continue;
        tc05::fence_after();
        float sc[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int q = 4 * qhalf + c;
          uint32_t v[32];
          tc05::tmem_ld32(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(a * kPreN + q * 32), v);
          tc05::tmem_ld_wait();
          float s = 0.f;
#pragma unroll
          for (int h = 0; h < 32; ++h) s = fmaf(bars.w[q][h], fmaxf(__uint_as_float(v[h]), 0.f), s);
          sc[c] = s;
        }
        tc05::fence_before();
        __syncwarp();
        if (lane == 0) tc05::mbar_arrive(&bars.tempty[a]);
        if (e == 0 && lane == 0) bars.drained = t_glob + 1;
        const long long j = (long long)t * kTileKeys + 32 * quarter + lane;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int q = 4 * qhalf + c, r = it.qt * kPreNQ + q;
          if (r < p.n_rows && j < p.N)
            p.scores[(size_t)r * p.scores_stride + j] = j < bars.nv[q] ? sc[c] : -INFINITY;
        }
      }
      // past the last tile of the query tile: -inf (done by the item holding the last tile)
      const PreItem last = pre_item(p, (it.qt + 1) * n_parts - 1, n_parts);
      if (it.t1 == last.t1) {
        const long long from = (long long)it.t1 * kTileKeys;
        for (int c = 0; c < kPreNQ; ++c) {
          const int r = it.qt * kPreNQ + c;
          if (r >= p.n_rows) break;
          for (long long jj = from + etid; jj < p.scores_len; jj += kPreEpiWarps * 32)
            p.scores[(size_t)r * p.scores_stride + jj] = -INFINITY;
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (bars.timeout && tid == 0) {
    for (int t = bars.consumed; t < bars.issued; ++t)
      tc05::mbar_wait(&bars.full[t % kPreStages], (t / kPreStages) & 1);
    for (int t = bars.drained; t < bars.consumed; ++t) tc05::mbar_wait(&bars.tfull[t & 1], (t >> 1) & 1);
    if (bars.q_issued > bars.q_used) tc05::mbar_wait(&bars.qfull, (bars.q_issued - 1) & 1);
  }
  __syncthreads();
  if (warp == 1) {
    tc05::fence_after();
    tc05::tmem_dealloc(tmem, kPreTmemCols);
  }
}

// ===================================================================================== host
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// Row-major [rows x 128] bf16 matrix, boxes of 64 columns x box_rows rows, 128-byte swizzle.
bool make_tmap(CUtensorMap* tm, const void* base, unsigned long long rows, unsigned box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {128, rows};
  const cuuint64_t strides[1] = {256};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major [rows x 128] byte matrix (FP8 keys), boxes of 128 columns x box_rows rows,
// 128-byte swizzle.
bool make_tmap_u8(CUtensorMap* tm, const void* base, unsigned long long rows, unsigned box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {128, rows};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t dec_smem_bytes(int K, int max_seg_blocks, bool fp8) {
  (void)K;
  return 1024 + (size_t)kDecRingBytes + (fp8 ? DecCfg<true>::kQBytes : DecCfg<false>::kQBytes) + sizeof(DecBars) +
         16 + sizeof(ArrSelShared) +
         (size_t)kDecSegMax * 4 + (size_t)max_seg_blocks * 4;
}

}  // namespace

bool mma_indexer_available() { return encode_fn() != nullptr; }

bool make_tmap_bf16(CUtensorMap* tm, const void* base, unsigned long long cols, unsigned long long rows,
                    unsigned long long row_bytes, unsigned box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int mma_decode_max_seg_blocks() { return 2048; }

int mma_decode_max_segment() { return kDecSegMax; }
// The segments of a row can run as one thread-block cluster (2..16 blocks, every cluster of
// the grid resident at once).
bool cluster_ok_query(int n_seg, int n_rows, int K, int max_seg_blocks, bool fp8);

bool mma_decode_cluster_ok(int n_seg, int n_rows, int K, int max_seg_blocks, bool fp8) {
  if (n_seg < 2 || n_seg > 16 || K > CSA2_MAX_TOPK) return false;
  // the answer depends on the device, the kernel and the launch shape only: remembered
  struct Entry {
    int dev, n_seg, n_rows, smem_key;
    bool fp8, ok;
  };
  static Entry cache[32];
  static int n_cache = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const int smem_key = (int)dec_smem_bytes(K, max_seg_blocks, fp8);
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_cache; ++i)
    if (cache[i].dev == dev && cache[i].n_seg == n_seg && cache[i].n_rows == n_rows && cache[i].smem_key == smem_key &&
        cache[i].fp8 == fp8)
      return cache[i].ok;
  const bool ok = cluster_ok_query(n_seg, n_rows, K, max_seg_blocks, fp8);
  cache[n_cache % 32] = Entry{dev, n_seg, n_rows, smem_key, fp8, ok};
  if (n_cache < 32) ++n_cache;
  return ok;
}

template <bool FP8>
bool cluster_ok_query_t(int n_seg, int n_rows, int K, int max_seg_blocks) {
  const size_t smem = dec_smem_bytes(K, max_seg_blocks, FP8);
  if (cudaFuncSetAttribute(idx_mma_decode_kernel<FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return false;
  if (n_seg > 8 &&
      cudaFuncSetAttribute(idx_mma_decode_kernel<FP8>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return false;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_seg, n_rows);
  cfg.blockDim = dim3(DecCfg<FP8>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)n_seg;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, idx_mma_decode_kernel<FP8>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return clusters >= n_rows;
}

bool cluster_ok_query(int n_seg, int n_rows, int K, int max_seg_blocks, bool fp8) {
  return fp8 ? cluster_ok_query_t<true>(n_seg, n_rows, K, max_seg_blocks)
             : cluster_ok_query_t<false>(n_seg, n_rows, K, max_seg_blocks);
}

bool mma_decode_can_merge(int n_seg, int K) { return n_seg <= 64 && (long long)n_seg * K <= kDecSegMax; }

size_t mma_decode_smem_bytes(int K, int max_seg_blocks, bool fp8) { return dec_smem_bytes(K, max_seg_blocks, fp8); }

template <bool FP8>
cudaError_t launch_mma_decode_t(const ScanParams& p, long long n_seq_rows, int n_seg, int max_seg_blocks,
                                cudaStream_t stream) {
  CUtensorMap tmK, tmQ, tmK64;
  const bool maps = FP8 ? make_tmap_u8(&tmK, p.k_idx, (unsigned long long)n_seq_rows, kTileKeys) &&
                              make_tmap_u8(&tmK64, p.k_idx, (unsigned long long)n_seq_rows, 64)
                        : make_tmap(&tmK, p.k_idx, (unsigned long long)n_seq_rows, kTileKeys) &&
                              make_tmap(&tmK64, p.k_idx, (unsigned long long)n_seq_rows, 64);
  if (!maps || !make_tmap(&tmQ, p.q_idx, (unsigned long long)p.n_rows * 32, 32)) return cudaErrorInvalidValue;
  ScanParams q = p;
  q.seg_table = max_seg_blocks;
  // the bitmap of marked entries follows the block table when it fits in shared memory
  q.fast_select = p.cluster_merge && p.K > 0 && dec_smem_bytes(p.K, max_seg_blocks, FP8) + kFastBytes <= 232448;
  const size_t smem = dec_smem_bytes(p.K, max_seg_blocks, FP8) + (q.fast_select ? kFastBytes : 0);
  auto kern = idx_mma_decode_kernel<FP8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  q.pdl_trigger = (long long)n_seg * p.n_rows <= device_sm_count();  // one CTA per SM: a single wave
  // Programmatic dependent launch: the blocks may become resident while the previous kernel
  // in the stream finishes; they wait for it before reading anything.
  cudaLaunchAttribute attr[2] = {};
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_seg, p.n_rows);
  cfg.blockDim = dim3(DecCfg<FP8>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.cluster_merge) {
    // the segments of a row form one cluster
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)n_seg;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
    if (n_seg > 8) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
  }
  e = cudaLaunchKernelEx(&cfg, kern, tmK, tmQ, tmK64, q);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_mma_decode(const ScanParams& p, long long n_seq_rows, int n_seg, int max_seg_blocks, bool fp8,
                              cudaStream_t stream) {
  if (p.n_rows == 0) return cudaSuccess;
  if (dec_smem_bytes(p.K, max_seg_blocks, fp8) > 232448) return cudaErrorInvalidValue;
  if (p.cand != nullptr && (p.cand_run <= 0 || p.cand_run % 64 != 0)) return cudaErrorInvalidValue;
  if (fp8 && p.k_scale == nullptr) return cudaErrorInvalidValue;
  return fp8 ? launch_mma_decode_t<true>(p, n_seq_rows, n_seg, max_seg_blocks, stream)
             : launch_mma_decode_t<false>(p, n_seq_rows, n_seg, max_seg_blocks, stream);
}

// FP8 streaming decode scan: usable for this K where two blocks fit on an SM.
bool fp8_stream_ok(int K) {
  if (K < 1 || K > kEngMaxK) return false;
  struct Entry {
    int dev, K;
    bool ok;
  };
  static Entry cache[16];
  static int n_cache = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_cache; ++i)
    if (cache[i].dev == dev && cache[i].K == K) return cache[i].ok;
  bool ok = false;
  const size_t smem = str_smem_bytes(K);
  // The occupancy query reports one block per SM for every kernel that allocates tensor memory
  // whatever its resources, so the fit of two blocks is checked here from the resources
  // themselves (tensor memory: two blocks of 256 of the SM's 512 columns).
  cudaFuncAttributes fa{};
  int smem_sm = 0, reserved = 0, regs_sm = 0;
  if (cudaFuncSetAttribute(idx_fp8_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) ==
          cudaSuccess &&
      cudaFuncSetAttribute(idx_fp8_stream_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared) == cudaSuccess &&
      cudaFuncGetAttributes(&fa, idx_fp8_stream_kernel) == cudaSuccess &&
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) == cudaSuccess) {
    const size_t block_smem = smem + fa.sharedSizeBytes + (size_t)reserved;
    const int warp_regs = (fa.numRegs * 32 + 255) / 256 * 256;  // allocated per warp in units of 256
    ok = 2 * block_smem <= (size_t)smem_sm && 2 * warp_regs * (kStrThreads / 32) <= regs_sm;
  }
  cudaGetLastError();
  cache[n_cache % 16] = Entry{dev, K, ok};
  if (n_cache < 16) ++n_cache;
  return ok;
}

cudaError_t launch_fp8_stream(const ScanParams& p, long long n_seq_rows, int n_seg, cudaStream_t stream) {
  if (p.n_rows == 0) return cudaSuccess;
  if (p.K < 1 || p.K > kEngMaxK || p.k_scale == nullptr || p.cand != nullptr || p.block_max != nullptr ||
      p.scores != nullptr || (n_seg > 1 && (p.seg_keys == nullptr || p.seg_pos == nullptr || p.seg_cnt == nullptr ||
                                            p.seg_thr == nullptr)))
    return cudaErrorInvalidValue;
  CUtensorMap tmK;
  if (!make_tmap_u8(&tmK, p.k_idx, (unsigned long long)n_seq_rows, kTileKeys)) return cudaErrorInvalidValue;
  const size_t smem = str_smem_bytes(p.K);
  cudaError_t e = cudaFuncSetAttribute(idx_fp8_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the set-up overlaps the previous kernel in the stream
  cudaLaunchAttribute attr[1] = {};
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_seg, p.n_rows);
  cfg.blockDim = dim3(kStrThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, idx_fp8_stream_kernel, tmK, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

size_t mma_prefill_smem_bytes() { return 1024 + (size_t)kPreStages * kKeyTile + 2 * kPreQHalf + sizeof(PreBars); }

cudaError_t launch_mma_prefill(const ScanParams& p, int n_ctas, int n_parts, cudaStream_t stream) {
  if (p.n_rows == 0) return cudaSuccess;
  CUtensorMap tmK, tmQ;
  if (!make_tmap(&tmK, p.k_idx, (unsigned long long)p.N, kTileKeys) ||
      !make_tmap(&tmQ, p.q_idx, (unsigned long long)p.n_rows * 32, kPreN))
    return cudaErrorInvalidValue;
  const int n_qt = (p.n_rows + kPreNQ - 1) / kPreNQ;
  const int n_items = n_qt * n_parts;
  const size_t smem = mma_prefill_smem_bytes();
  cudaError_t e =
      cudaFuncSetAttribute(idx_mma_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  idx_mma_prefill_kernel<<<n_ctas < n_items ? n_ctas : n_items, kPreThreads, smem, stream>>>(tmK, tmQ, p, n_items,
                                                                                            n_parts);
  return cudaGetLastError();
}

}  // namespace csa2
