// Lightning-indexer scan for decode rows: score_j = sum_h w_h * ReLU(q^I_h . k^I_j)
// ("Every layer, connected", "The global and index paths"), fused with the causal mask,
// block maxima for the hierarchical pool and an exact per-segment top-K.
//
// One thread block (16 warps) handles one segment of one query row.  Each warp streams its
// own contiguous range of 16-record tiles through a private cp.async ring in shared memory
// (every thread reads back only the bytes it copied, so no block barrier is needed in the
// hot loop) and multiplies them on the tensor cores with warp-level bf16 MMA:
//   M = 16 records, N = 8 indexer heads (x4 tiles = 32 heads), K = 128 dims (8 steps).
// The indexer query is held in registers as B fragments for the whole scan.  The 128 dims
// are consumed in a permuted order chosen so that each thread's 16-byte copies are the
// exact A-fragment words it needs; q uses the same permutation, so the dot products are
// unchanged.  FP8 keys are widened to f16 in registers by one hardware conversion per pair
// (exact) and meet q^I widened once to f16 (exact for every element within ~2^-38 of its
// head's largest: each head is scaled by the power of two that puts its largest element in
// [2^14, 2^15), the inverse factor going into the head weight); the record's row scale is
// applied to each head's dot product before the ReLU.
#include "select.cuh"
#include "kernels.h"

namespace csa2 {

namespace {

constexpr int kScanWarps = 16;
constexpr int kScanThreads = kScanWarps * 32;
constexpr int kRoundTiles = kRoundEntries / 16;  // 8 tiles of 16 records between checks

// Key formats of the scan: bf16 rows, FP8 E4M3 rows with an fp32 scale, OCP MXFP4 rows
// (E2M1 codes, one UE8M0 exponent per block of 32; the pages' indexer precision).
enum { kKeyBF16 = 0, kKeyFP8 = 1, kKeyMX = 2 };

template <int FMT>
struct ScanCfg {
  static constexpr int kRowBytes = FMT == kKeyBF16 ? 256 : FMT == kKeyFP8 ? 128 : 64;  // one indexer key
  // one 16-record tile; MXFP4: the records' four exponent bytes follow the codes
  static constexpr int kStageBytes = 16 * kRowBytes + (FMT == kKeyMX ? 64 : 0);
  static constexpr int kStages = FMT == kKeyBF16 ? 2 : FMT == kKeyFP8 ? 4 : 6;
  static constexpr int kRingBytes = kScanWarps * kStages * kStageBytes;
};

// Index (in 32-bit words of a 128-dim bf16 row) of the q^I pair that meets A-fragment word
// `hi` (0 = k-lo pair, 1 = k-hi pair) of k-step s for the thread with c = lane % 4.
template <int FMT>
__device__ __forceinline__ int q_word(int s, int c, int hi) {
  if (FMT == kKeyMX) {
    // 16-byte chunk c of the 64-byte MXFP4 row is block c (dims 32c .. 32c+31, two per
    // byte); k-step s uses its bytes 2s (dims 32c + 4s + {0,1}) and 2s+1 ({2,3})
    return 16 * c + 2 * s + hi;
  }
  if (FMT == kKeyFP8) {
    // 16-byte chunk (4*(s/4) + c) of the 128-byte FP8 row holds 16 dims; k-step s uses its
    // word s%4: dims 16*chunk + 4*(s%4) + {0,1} (lo) and {2,3} (hi).
    const int chunk = 4 * (s >> 2) + c;
    return 8 * chunk + 2 * (s & 3) + hi;
  } else {
    // 16-byte chunk u = 4*(s/2) + c of the 256-byte bf16 row holds 8 dims; k-step s uses
    // dims 8u + 4*(s%2) + {0,1} (lo) and {2,3} (hi).
    const int u = 4 * (s >> 1) + c;
    return 4 * u + 2 * (s & 1) + hi;
  }
}

template <int FMT, bool GATHER>
__global__ void __launch_bounds__(kScanThreads, 1) index_scan_kernel(const ScanParams p) {
  constexpr bool FP8 = FMT == kKeyFP8, MX = FMT == kKeyMX, WIDE = FMT != kKeyBF16;  // WIDE: f16 MMA
  using Cfg = ScanCfg<FMT>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  Engine<kScanWarps> eng;
  eng.sh = reinterpret_cast<EngShared*>(smem + Cfg::kRingBytes);
  eng.cap = p.K + kRoundEntries;
  eng.keys = reinterpret_cast<uint32_t*>(smem + Cfg::kRingBytes + sizeof(EngShared));
  eng.js = reinterpret_cast<int32_t*>(eng.keys + kScanWarps * eng.cap);
  eng.out_key = reinterpret_cast<uint32_t*>(eng.js + kScanWarps * eng.cap);
  eng.out_j = reinterpret_cast<int32_t*>(eng.out_key + p.K);
  eng.bar_id = 0;
  eng.tid = threadIdx.x;

  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int row = blockIdx.y, seg = blockIdx.x, n_seg = gridDim.x;
  const int b = p.seq_of_row[row];
  const long long L_row = GATHER ? min((long long)p.n_cand[row], p.cand_stride)
                                  : min((long long)p.n_visible[row], p.N);

  // ---- this warp's entry range: units of U entries split over segments, then warps
  const int U = p.unit;
  const long long n_units = (L_row + U - 1) / U;
  long long u0, u1, w0, w1;
  split_range(n_units, n_seg, seg, u0, u1);
  split_range(u1 - u0, kScanWarps, wid, w0, w1);
  const long long e0 = (u0 + w0) * U;
  const long long e1 = min((u0 + w1) * U, L_row);
  const long long tb = e0 / 16, te = (e1 + 15) / 16;

  // ---- indexer query as B fragments, weights for this thread's heads
  uint32_t qf[8][4][2];
  {
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(p.q_idx) + (size_t)row * kIdxHeads * (kIdxDim / 2);
#pragma unroll
    for (int s = 0; s < 8; ++s)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const uint32_t* qh = qrow + (8 * nt + g) * (kIdxDim / 2);
        qf[s][nt][0] = __ldg(qh + q_word<FMT>(s, c, 0));
        qf[s][nt][1] = __ldg(qh + q_word<FMT>(s, c, 1));
      }
  }
  float wv[4][2];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    wv[nt][0] = __ldg(p.w + (size_t)row * kIdxHeads + 8 * nt + 2 * c);
    wv[nt][1] = __ldg(p.w + (size_t)row * kIdxHeads + 8 * nt + 2 * c + 1);
  }
  if (WIDE) {
    // q^I to f16: the four lanes of a group hold head 8nt+g's 128 dims between them
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      uint32_t mx = 0u;
#pragma unroll
      for (int s = 0; s < 8; ++s)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) mx = max(mx, max(qf[s][nt][h2] & 0x7fffu, (qf[s][nt][h2] >> 16) & 0x7fffu));
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const int ex = (int)((mx >> 7) & 0xffu) - 127;
      const int e = mx == 0u ? 0 : min(126, max(-126, 14 - ex));
      const float f = __int_as_float((e + 127) << 23);
#pragma unroll
      for (int s = 0; s < 8; ++s)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const uint32_t v = qf[s][nt][h2];
          const __half2 hv = __floats2half2_rn(__uint_as_float(v << 16) * f, __uint_as_float(v & 0xffff0000u) * f);
          qf[s][nt][h2] = *reinterpret_cast<const uint32_t*>(&hv);
        }
      // this lane's accumulator columns are heads 8nt+2c and 8nt+2c+1 (groups 2c, 2c+1)
      const int e0 = __shfl_sync(0xffffffffu, e, 8 * c), e1 = __shfl_sync(0xffffffffu, e, 8 * c + 4);
      wv[nt][0] *= __int_as_float((127 - e0) << 23);
      wv[nt][1] *= __int_as_float((127 - e1) << 23);
    }
  }

  const uint8_t* kbase = reinterpret_cast<const uint8_t*>(p.k_idx);
  const size_t seq_off = (size_t)b * (size_t)p.N;
  uint8_t* my_ring = ring + (size_t)wid * Cfg::kStages * Cfg::kStageBytes;

  auto record_of = [&](long long j) -> long long {
    if (GATHER) return (long long)__ldg(p.cand + (size_t)row * p.cand_stride + j);
    return j;
  };
  // Issues the copies of tile t into its ring stage (zero-fill past the warp's range).
  auto issue = [&](long long t) {
    uint8_t* st = my_ring + (int)(t % Cfg::kStages) * Cfg::kStageBytes;
#pragma unroll
    for (int rh = 0; rh < 2; ++rh) {
      const long long j = t * 16 + g + 8 * rh;
      const bool valid = j < e1;
      const long long rec = valid ? record_of(j) : 0;
      const uint8_t* src = kbase + (seq_off + (size_t)rec) * Cfg::kRowBytes;
      if (MX) {
        // chunk c (block c) of the row; lane c = 0 of each group also copies the row's
        // four exponent bytes
        cp_async16(st + rh * 512 + lane * 16, src + c * 16, valid);
        if (c == 0)
          cp_async4(st + 1024 + (g + 8 * rh) * 4,
                    reinterpret_cast<const uint8_t*>(p.k_scale) + (seq_off + (size_t)rec) * 4, valid);
      } else if (FP8) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
          cp_async16(st + (2 * i + rh) * 512 + lane * 16, src + (4 * i + c) * 16, valid);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          cp_async16(st + (2 * i + rh) * 512 + lane * 16, src + (4 * i + c) * 16, valid);
      }
    }
  };

  const bool do_topk = p.K > 0;
  if (do_topk) eng_init(eng);
  int cnt = 0;
  uint32_t thr = 0u;

  // rounds: every warp runs the same number so that the block can meet between rounds
  const long long max_tiles_w = ((u1 - u0 + kScanWarps - 1) / kScanWarps) * (U / 16) + 1;
  const int rounds = (int)((max_tiles_w + kRoundTiles - 1) / kRoundTiles);

#pragma unroll
  for (int k = 0; k < Cfg::kStages - 1; ++k) {
    if (tb + k < te) issue(tb + k);
    cp_async_commit();
  }

  float bmax = -INFINITY;  // running block max (warp-uniform)
  long long t = tb;
  for (int r = 0; r < rounds; ++r) {
    for (int k = 0; k < kRoundTiles; ++k, ++t) {
      if (t < te) {
        if (t + Cfg::kStages - 1 < te) issue(t + Cfg::kStages - 1);
        cp_async_commit();
        cp_async_wait<Cfg::kStages - 1>();
        const uint8_t* st = my_ring + (int)(t % Cfg::kStages) * Cfg::kStageBytes;
        float acc[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        if (MX) {
          // the row's largest block exponent E scales the dot product (below); block c's
          // codes take 2^(e_c - E) in f16 (exact while e_c - E >= -23)
          const uint4 r0 = *reinterpret_cast<const uint4*>(st + lane * 16);
          const uint4 r1 = *reinterpret_cast<const uint4*>(st + 512 + lane * 16);
          const uint32_t x0 = *reinterpret_cast<const uint32_t*>(st + 1024 + g * 4);
          const uint32_t x1 = *reinterpret_cast<const uint32_t*>(st + 1024 + (g + 8) * 4);
          auto block_factor = [&](uint32_t x) -> __half2 {
            const uint32_t e0 = x & 0xffu, e1 = (x >> 8) & 0xffu, e2 = (x >> 16) & 0xffu, e3 = x >> 24;
            const int E = (int)max(max(e0, e1), max(e2, e3));
            const int d = (int)((x >> (8 * c)) & 0xffu) - E;  // <= 0
            const float f = d < -126 ? 0.f : __int_as_float((d + 127) << 23);
            return __float2half2_rn(f);
          };
          const __half2 f0 = block_factor(x0), f1 = block_factor(x1);
          const uint32_t w0v[4] = {r0.x, r0.y, r0.z, r0.w};
          const uint32_t w1v[4] = {r1.x, r1.y, r1.z, r1.w};
#pragma unroll
          for (int s = 0; s < 8; ++s) {
            const uint32_t b0 = (w0v[s >> 1] >> (16 * (s & 1))) & 0xffffu;  // bytes 2s, 2s+1 of row g
            const uint32_t b1 = (w1v[s >> 1] >> (16 * (s & 1))) & 0xffffu;  // ... of row g+8
            auto wid = [](uint32_t byte, __half2 f) -> uint32_t {
              uint32_t h = e2m1x2_to_f16x2(byte);
              __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&h), f);
              return *reinterpret_cast<const uint32_t*>(&v);
            };
            const uint32_t a0 = wid(b0 & 0xffu, f0), a2 = wid(b0 >> 8, f0);
            const uint32_t a1 = wid(b1 & 0xffu, f1), a3 = wid(b1 >> 8, f1);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) mma_f16(acc[nt], a0, a1, a2, a3, qf[s][nt][0], qf[s][nt][1]);
          }
        } else if (FP8) {
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const uint4 r0 = *reinterpret_cast<const uint4*>(st + (2 * i) * 512 + lane * 16);
            const uint4 r1 = *reinterpret_cast<const uint4*>(st + (2 * i + 1) * 512 + lane * 16);
            const uint32_t w0v[4] = {r0.x, r0.y, r0.z, r0.w};
            const uint32_t w1v[4] = {r1.x, r1.y, r1.z, r1.w};
#pragma unroll
            for (int jw = 0; jw < 4; ++jw) {
              const int s = 4 * i + jw;
              const uint32_t a0 = e4m3x2_to_f16x2((uint16_t)(w0v[jw] & 0xffffu));
              const uint32_t a2 = e4m3x2_to_f16x2((uint16_t)(w0v[jw] >> 16));
              const uint32_t a1 = e4m3x2_to_f16x2((uint16_t)(w1v[jw] & 0xffffu));
              const uint32_t a3 = e4m3x2_to_f16x2((uint16_t)(w1v[jw] >> 16));
#pragma unroll
              for (int nt = 0; nt < 4; ++nt) mma_f16(acc[nt], a0, a1, a2, a3, qf[s][nt][0], qf[s][nt][1]);
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 r0 = *reinterpret_cast<const uint4*>(st + (2 * i) * 512 + lane * 16);
            const uint4 r1 = *reinterpret_cast<const uint4*>(st + (2 * i + 1) * 512 + lane * 16);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
              mma_bf16(acc[nt], r0.x, r1.x, r0.y, r1.y, qf[2 * i][nt][0], qf[2 * i][nt][1]);
              mma_bf16(acc[nt], r0.z, r1.z, r0.w, r1.w, qf[2 * i + 1][nt][0], qf[2 * i + 1][nt][1]);
            }
          }
        }
        // ---- epilogue: ReLU, head weights, sum over the 32 heads
        const long long j_lo = t * 16 + g, j_hi = j_lo + 8;
        const bool v_lo = j_lo < e1, v_hi = j_hi < e1;
        float sc_lo = 1.f, sc_hi = 1.f;
        long long rec_lo = j_lo, rec_hi = j_hi;
        if (GATHER || FP8) {
          rec_lo = v_lo ? record_of(j_lo) : 0;
          rec_hi = v_hi ? record_of(j_hi) : 0;
        }
        if (FP8) {
          sc_lo = __ldg(p.k_scale + seq_off + rec_lo);
          sc_hi = __ldg(p.k_scale + seq_off + rec_hi);
        }
        if (MX) {
          // 2^(E - 127) of the row's largest block exponent E (from the stage)
          auto row_scale = [](uint32_t x) -> float {
            const uint32_t E = max(max(x & 0xffu, (x >> 8) & 0xffu), max((x >> 16) & 0xffu, x >> 24));
            return E == 0u ? __int_as_float(1 << 22) : __int_as_float((int)E << 23);  // 2^(E-127), exact
          };
          const uint8_t* st = my_ring + (int)(t % Cfg::kStages) * Cfg::kStageBytes;
          sc_lo = row_scale(*reinterpret_cast<const uint32_t*>(st + 1024 + g * 4));
          sc_hi = row_scale(*reinterpret_cast<const uint32_t*>(st + 1024 + (g + 8) * 4));
        }
        float s_lo = 0.f, s_hi = 0.f;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          if (WIDE) {
            s_lo = fmaf(wv[nt][0], fmaxf(acc[nt][0] * sc_lo, 0.f), s_lo);
            s_lo = fmaf(wv[nt][1], fmaxf(acc[nt][1] * sc_lo, 0.f), s_lo);
            s_hi = fmaf(wv[nt][0], fmaxf(acc[nt][2] * sc_hi, 0.f), s_hi);
            s_hi = fmaf(wv[nt][1], fmaxf(acc[nt][3] * sc_hi, 0.f), s_hi);
          } else {
            s_lo = fmaf(wv[nt][0], fmaxf(acc[nt][0], 0.f), s_lo);
            s_lo = fmaf(wv[nt][1], fmaxf(acc[nt][1], 0.f), s_lo);
            s_hi = fmaf(wv[nt][0], fmaxf(acc[nt][2], 0.f), s_hi);
            s_hi = fmaf(wv[nt][1], fmaxf(acc[nt][3], 0.f), s_hi);
          }
        }
        s_lo += __shfl_xor_sync(0xffffffffu, s_lo, 1);
        s_lo += __shfl_xor_sync(0xffffffffu, s_lo, 2);
        s_hi += __shfl_xor_sync(0xffffffffu, s_hi, 1);
        s_hi += __shfl_xor_sync(0xffffffffu, s_hi, 2);

        if (p.scores != nullptr && c == 0) {
          float* so = p.scores + (size_t)row * p.scores_stride;
          if (v_lo) so[j_lo] = s_lo;
          if (v_hi) so[j_hi] = s_hi;
        }
        if (p.block_max != nullptr) {
          // U == block_size here, so a block is bs/16 consecutive tiles of this warp
          bmax = fmaxf(bmax, warp_max(fmaxf(v_lo ? s_lo : -INFINITY, v_hi ? s_hi : -INFINITY)));
          const long long tile_end = t * 16 + 16;
          if (tile_end % U == 0 || t + 1 == te) {
            if (lane == 0) p.block_max[(size_t)row * p.bmax_stride + (t * 16) / U] = bmax;
            bmax = -INFINITY;
          }
        }
        if (do_topk) {
          eng_append(eng, cnt, thr, c == 0 && v_lo, score_key(s_lo), (int32_t)j_lo);
          eng_append(eng, cnt, thr, c == 0 && v_hi, score_key(s_hi), (int32_t)j_hi);
        }
      }
    }
    if (do_topk) thr = eng_check(eng, p.K, cnt);
  }
  cp_async_wait<0>();

  // ---- entries past the candidates: -inf scores and empty blocks (last segment only)
  if (seg == n_seg - 1) {
    if (p.scores != nullptr)
      for (long long j = L_row + tid; j < p.scores_len; j += kScanThreads)
        p.scores[(size_t)row * p.scores_stride + j] = -INFINITY;
    if (p.block_max != nullptr)
      for (long long blk = (L_row + U - 1) / U + tid; blk < p.n_blocks; blk += kScanThreads)
        p.block_max[(size_t)row * p.bmax_stride + blk] = -INFINITY;
  }
  if (!do_topk) return;
  uint32_t* thr_out = n_seg > 1 ? p.seg_thr + (size_t)row * n_seg + seg : nullptr;
  const int n = eng_finish(eng, p.K, cnt, thr_out);
  if (n_seg == 1) {
    int32_t* out = p.idx + (size_t)row * p.K;
    for (int i = tid; i < p.K; i += kScanThreads) out[i] = i < n ? (int32_t)record_of(eng.out_j[i]) : -1;
  } else {
    const size_t o = ((size_t)row * n_seg + seg) * p.K;
    for (int i = tid; i < n; i += kScanThreads) {
      p.seg_keys[o + i] = eng.out_key[i];
      p.seg_pos[o + i] = (int32_t)record_of(eng.out_j[i]);
    }
    if (tid == 0) p.seg_cnt[(size_t)row * n_seg + seg] = n;
  }
}

}  // namespace

size_t scan_smem_bytes(int fmt, int K) {
  const size_t ring = fmt == kKeyFP8 ? ScanCfg<kKeyFP8>::kRingBytes
                      : fmt == kKeyMX ? ScanCfg<kKeyMX>::kRingBytes
                                      : ScanCfg<kKeyBF16>::kRingBytes;
  size_t s = ring + sizeof(EngShared);
  if (K > 0) s += (size_t)kScanWarps * (K + kRoundEntries) * 8 + (size_t)K * 8;
  return s;
}

cudaError_t launch_index_scan(const ScanParams& p, int fmt, bool gather, int n_seg, cudaStream_t stream) {
  const size_t smem = scan_smem_bytes(fmt, p.K);
  dim3 grid(n_seg, p.n_rows), block(kScanThreads);
  if (p.n_rows == 0) return cudaSuccess;
#define CSA2_LAUNCH_SCAN(F, G)                                                                         \
  do {                                                                                                 \
    cudaError_t e = cudaFuncSetAttribute(index_scan_kernel<F, G>,                                      \
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);      \
    if (e != cudaSuccess) return e;                                                                    \
    index_scan_kernel<F, G><<<grid, block, smem, stream>>>(p);                                         \
  } while (0)
  if (fmt == kKeyFP8) {
    if (gather) CSA2_LAUNCH_SCAN(kKeyFP8, true); else CSA2_LAUNCH_SCAN(kKeyFP8, false);
  } else if (fmt == kKeyMX) {
    if (gather) CSA2_LAUNCH_SCAN(kKeyMX, true); else CSA2_LAUNCH_SCAN(kKeyMX, false);
  } else {
    if (gather) CSA2_LAUNCH_SCAN(kKeyBF16, true); else CSA2_LAUNCH_SCAN(kKeyBF16, false);
  }
#undef CSA2_LAUNCH_SCAN
  return cudaGetLastError();
}

}  // namespace csa2
