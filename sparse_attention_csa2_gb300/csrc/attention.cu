// Sparse shared-latent MQA of one query row over its selected latents plus its sliding
// window, with one sink logit per head ("DeepSeek V4 Inside", CSA core attention and
// eq. (27); "Every layer, connected", "The query and output paths").
//
// The K + W attended entries of a row are cut into tiles of 128; one thread block takes one
// tile of one row for all 64 heads, on the fifth-generation tensor cores:
//   gather   the tile's 128 latent rows (bf16 by cp.async; FP4 latents and FP8 window rows
//            widened to bf16 in registers, which is exact) and the row's query q' = RoPE(q)
//            into shared memory, both in the 128-byte-swizzled K-major layout;
//   S^T      = K q'^T: M = 128 entries x N = 64 heads x K = 512, bf16 in, fp32 in TMEM; the
//            rotated dims of q' enter as two bf16 terms (hi + lo, four more K-steps against
//            the tile's rotary panel), so only the stored latents and query are bf16;
//   softmax  one thread per entry reads its 64 logits from TMEM, scales them (FP8 window
//            rows: times their row scale), and the tile's per-head maximum M_h and sum l_h
//            are reduced over the 128 entries; P = exp(S - M) is written back to shared
//            memory as two bf16 terms P = P_hi + P_lo (about 16 significant bits; FP8 rows'
//            weights times their row scale);
//   O^T      = V^T P^T with V = the same latent tile read transposed (MN-major operand):
//            four M = 128-dim chunks x N = 128 (P_hi and P_lo side by side, 64 heads each)
//            x K = 128 entries, fp32 in TMEM (the two halves are added when read out);
//   partial  (M_h, l_h, O) of the tile go to the workspace.
// A second kernel merges a row's tiles (log-sum-exp), adds the sink to the denominator,
// normalises and turns the output's rotary coordinates back by -position.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "kernels.h"
#include "tc05.cuh"

namespace csa2 {

namespace {

constexpr int kAttnThreads = 256;                  // 8 warps
constexpr int kTileE = 128;                        // attended entries per block (MMA M)
constexpr int kQPanel = kHeads * 128;              // 8 KB: 64 heads x 64 dims (bf16)
constexpr int kKPanel = kTileE * 128;              // 16 KB: 128 entries x 64 dims
// q' in eight panels, then the low bf16 parts of its rotary dims (448..511) as a ninth; P_hi,
// P_lo after the first GEMM
constexpr int kQBytes = 9 * kQPanel;               // 72 KB
constexpr int kKBytes = 8 * kKPanel;               // 128 KB
constexpr int kPBytes = kTileE * 128;              // 16 KB: 128 entries x 64 heads (bf16)

struct TileSrc {
  const uint8_t* ptr[kTileE];   // first byte of each entry's row (codes for FP formats)
  const uint8_t* sptr[kTileE];  // FP4 group scales
  float rs[kTileE];             // FP8 row scale (1 otherwise)
  int fmt[kTileE];              // storage format, -1 = masked entry
};

struct AttnShared {
  TileSrc src;
  float red[4][kHeads];      // per TMEM lane quarter: the per-head maximum over its 32 entries
  float red_sum[4][kHeads];  // ... and the per-head sum of P
  float mfin[kHeads];    // the tile's per-head maximum logit
  float cs[kRopeDim];    // cos (0..31) and sin (32..63) of the row's rotary angles
  uint64_t bar_s, bar_o;  // first and second GEMM completed
  uint32_t tmem_base;
  int timeout;
  int s_issued, o_issued;
};
constexpr int kAttnSmemBytes = 1024 + kQBytes + kKBytes + (int)sizeof(AttnShared);

__device__ __forceinline__ uint8_t* align_1k(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

// Byte offset of 16-byte chunk c (dims 8c .. 8c+7) of row r in a tile stored as eight
// 64-dim panels of `rows` rows x 128 bytes, the 16-byte chunks of each row XOR-ed with the
// row's low three bits (the tensor cores' 128-byte swizzle).
__device__ __forceinline__ int sw128_off(int r, int c, int rows) {
  return (c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// Shared-memory descriptor of a 128-byte-swizzled operand with explicit leading and stride
// byte offsets (MN-major operands: leading = distance between 64-element chunks along M or N,
// stride = distance between groups of 8 rows along K).
__device__ __forceinline__ uint64_t sw128_desc_lbo(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3ffffu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3fffu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3fffu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Two E4M3 codes (low byte first) -> two floats, exact (every E4M3 value is an f16 value).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint16_t v) {
  uint32_t h;
  asm("{\n .reg .b32 t;\n cvt.rn.f16x2.e4m3x2 t, %1;\n mov.b32 %0, t;\n}\n" : "=r"(h) : "h"(v));
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}
// Two E2M1 codes in one byte (low nibble first) -> two floats, exact.
__device__ __forceinline__ float2 e2m1x2_to_f32x2(uint32_t byte) {
  uint32_t h;
  asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}\n" : "=r"(h) : "r"(byte));
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}

// cos and sin of the rotary angle sign * pos * inv_freq.  The angle (up to ~2^31 rad) is
// formed and reduced modulo 2*pi in double (Cody-Waite with a two-part 2*pi), then the
// reduced angle (|r| <= pi) goes through single-precision sincosf.
__device__ __forceinline__ void rope_cs(long long pos, double inv_freq, float sign, float* c, float* s) {
  const double a = (double)pos * inv_freq;
  const double k = rint(a * 0.15915494309189535);  // 1 / (2 pi)
  double r = fma(-k, 6.283185307179586, a);
  r = fma(-k, 2.4492935982947064e-16, r);
  sincosf(sign * (float)r, s, c);
}

// Rotary cos/sin table of one position: cs[i] = cos, cs[32 + i] = sin.
__device__ __forceinline__ void rope_table(float* cs, const AttnParams& p, long long pos, float sign) {
  if (threadIdx.x < kRopeDim / 2) {
    const int i = threadIdx.x;
    rope_cs(pos, p.inv_freq[i], sign, &cs[i], &cs[kRopeDim / 2 + i]);
  }
}

struct EntrySrc {
  const uint8_t* ptr;   // first byte of the row (codes for FP formats)
  const uint8_t* sptr;  // FP4 group scales
  float rs;             // FP8 row scale
  int fmt;              // CSA2_BF16, CSA2_FP4_*, CSA2_FP8_E4M3_ROWSCALE
  bool valid;
};

// Entry e of a row's attended list: e < K are the selected latents (idx; -1 = none), then
// the window rows of positions lo .. qp.
__device__ __forceinline__ EntrySrc entry_source(const AttnParams& p, int row, int b, long long qp, long long lo,
                                                 long long pos0, int e) {
  EntrySrc s{nullptr, nullptr, 1.f, CSA2_BF16, false};
  if (e < p.K) {
    int rec = __ldg(p.idx + (size_t)row * p.K + e);
    if (p.range_count > 0 && rec >= 0) {  // another device's record, or this device's
      rec = (rec < p.range_first || rec >= p.range_first + p.range_count) ? -1 : (int)(rec - p.range_first);
    }
    if (rec < -1 || rec >= p.N) {
      if (p.dev_status != nullptr) atomicExch(p.dev_status, (int)CSA2_EDEVICE_INDEX);
    } else if (rec >= 0) {
      s.valid = true;
      s.fmt = p.lat_fmt;
      const size_t r = (size_t)b * (size_t)p.N + (size_t)rec;
      if (p.lat_fmt == CSA2_BF16) {
        s.ptr = reinterpret_cast<const uint8_t*>(p.lat) + r * 1024;
      } else {
        const int g = p.lat_fmt == CSA2_FP4_E2M1_G32 ? 32 : 16;
        s.ptr = reinterpret_cast<const uint8_t*>(p.lat) + r * 256;
        s.sptr = p.lat_scale + r * (kHeadDim / g);
      }
    }
  } else if (e < p.K + p.window && !p.skip_window) {
    const long long pos = lo + (e - p.K);
    if (pos <= qp && pos - pos0 < p.swa_rows) {
      s.valid = true;
      s.fmt = p.swa_fmt;
      const size_t r = (size_t)b * (size_t)p.swa_rows + (size_t)(pos - pos0);
      if (p.swa_fmt == CSA2_BF16) {
        s.ptr = reinterpret_cast<const uint8_t*>(p.swa) + r * 1024;
      } else {
        s.ptr = reinterpret_cast<const uint8_t*>(p.swa) + r * 512;
        s.rs = __ldg(p.swa_scale + r);
      }
    }
  }
  return s;
}

// Gathers the block's tile (128 entries x 512 dims, bf16, panel layout) into `ks`.  bf16 rows
// go by cp.async, a warp copying 512 contiguous bytes per instruction (masked entries are
// zero-filled, so they add nothing to P V); FP4 latents and FP8 window rows are widened to
// bf16 in registers (exact), two threads per row.
__device__ __forceinline__ void gather_tile(const TileSrc& m, uint8_t* ks, const void* any_valid) {
  const int t = threadIdx.x;
#pragma unroll 4
  for (int k = 0; k < kTileE / 4; ++k) {
    const int r = 4 * k + (t >> 6), c = t & 63;
    const int f = m.fmt[r];
    if (f == CSA2_BF16 || f < 0) {
      const uint8_t* src = f < 0 ? reinterpret_cast<const uint8_t*>(any_valid) : m.ptr[r];
      cp_async16(ks + sw128_off(r, c, kTileE), src + c * 16, f >= 0);
    }
  }
  const int r = t >> 1, half = t & 1;  // 256 dims per thread
  const int f = m.fmt[r];
  if (f == CSA2_FP8_E4M3_ROWSCALE) {
#pragma unroll 1
    for (int g = 0; g < 4; ++g) {
      const int d0 = half * 256 + g * 64;
      const uint4* src = reinterpret_cast<const uint4*>(m.ptr[r] + d0);
      uint32_t outw[32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint4 v = __ldg(src + q4);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          outw[q4 * 8 + 2 * k] = e4m3x2_to_bf16x2((uint16_t)(w4[k] & 0xffffu));
          outw[q4 * 8 + 2 * k + 1] = e4m3x2_to_bf16x2((uint16_t)(w4[k] >> 16));
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k)
        *reinterpret_cast<uint4*>(ks + sw128_off(r, d0 / 8 + k, kTileE)) =
            make_uint4(outw[4 * k], outw[4 * k + 1], outw[4 * k + 2], outw[4 * k + 3]);
    }
  } else if (f == CSA2_FP4_E2M1_G32 || f == CSA2_FP4_E2M1_G16) {
    // This thread's 256 dims use 8 (groups of 32) or 16 (groups of 16) E4M3 scale bytes,
    // loaded once; codes and scales are widened by the hardware conversions (E2M1 pair -> f16
    // pair, E4M3 pair -> f16 pair, both exact) and each product level x scale (at most 6
    // significant bits) is exact in bf16.
    const bool g16 = f == CSA2_FP4_E2M1_G16;
    uint4 sv;
    if (g16) {
      sv = __ldg(reinterpret_cast<const uint4*>(m.sptr[r] + half * 16));
    } else {
      const uint2 t2 = __ldg(reinterpret_cast<const uint2*>(m.sptr[r] + half * 8));
      sv = make_uint4(t2.x, t2.y, 0u, 0u);
    }
#pragma unroll 1
    for (int g = 0; g < 4; ++g) {
      const int d0 = half * 256 + g * 64;
      // the scales of dims d0 .. d0+63: four bytes (groups of 16) or two (groups of 32)
      const uint32_t sw = g16 ? (g == 0 ? sv.x : g == 1 ? sv.y : g == 2 ? sv.z : sv.w)
                              : ((g < 2 ? sv.x : sv.y) >> (16 * (g & 1))) & 0xffffu;
      const float2 s01 = e4m3x2_to_f32x2((uint16_t)(sw & 0xffffu));
      const float2 s23 = e4m3x2_to_f32x2((uint16_t)(sw >> 16));
      const float sc[4] = {s01.x, s01.y, s23.x, s23.y};
      const uint4* src = reinterpret_cast<const uint4*>(m.ptr[r] + d0 / 2);
      uint32_t outw[32];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const uint4 v = __ldg(src + h2);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
#pragma unroll
          for (int byte = 0; byte < 4; ++byte) {
            const int lc = h2 * 32 + k * 8 + byte * 2;  // even channel of this byte within the 64
            const float s = sc[g16 ? lc / 16 : lc / 32];
            const float2 lv = e2m1x2_to_f32x2((w4[k] >> (8 * byte)) & 0xffu);
            outw[h2 * 16 + k * 4 + byte] = pack_bf16x2(lv.x * s, lv.y * s);
          }
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k)
        *reinterpret_cast<uint4*>(ks + sw128_off(r, d0 / 8 + k, kTileE)) =
            make_uint4(outw[4 * k], outw[4 * k + 1], outw[4 * k + 2], outw[4 * k + 3]);
    }
  }
}

// Heads h0 .. h0+NH-1 of the row's query (NH x 512 dims) into `qs` (panel layout, NH rows per
// 64-dim panel) by cp.async, one 16-byte chunk per copy (consecutive threads on consecutive
// chunks); rotate_query then turns the rotary pairs (dims 448 + 2i, 448 + 2i + 1) in place once
// the copies have landed.
template <int NH>
__device__ __forceinline__ void copy_query(const AttnParams& p, int row, int h0, uint8_t* qs) {
  const uint8_t* qsrc = reinterpret_cast<const uint8_t*>(p.q) + ((size_t)row * kHeads + h0) * kHeadDim * 2;
#pragma unroll 1  // run-once code: kept small for the instruction cache (measured)
  for (int k = 0; k < NH * kHeadDim / 8 / kAttnThreads; ++k) {
    const int idx = k * kAttnThreads + threadIdx.x, h = idx >> 6, ch = idx & 63;
    cp_async16(qs + sw128_off(h, ch, NH), qsrc + (size_t)idx * 16, true);
  }
}
// The rotated coordinates go to the tensor cores as two bf16 terms, hi = bf16(x') in panel 7
// and lo = bf16(x' - hi) in panel 8 (a ninth K-panel of the first GEMM), so the logits see x'
// to ~2^-16 instead of bf16's 2^-8: with peaked attention that rounding was the largest error
// of the output.
template <int NH>
__device__ __forceinline__ void rotate_query(uint8_t* qs, const float* cs) {
#pragma unroll 1  // run-once code: kept small for the instruction cache (measured)
  for (int idx = threadIdx.x; idx < NH * 8; idx += kAttnThreads) {
    const int h = idx >> 3, ch = 56 + (idx & 7);
    uint4* q4 = reinterpret_cast<uint4*>(qs + sw128_off(h, ch, NH));
    const uint4 v = *q4;
    uint32_t w4[4] = {v.x, v.y, v.z, v.w}, lo4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = (ch - 56) * 4 + j;  // rotary pair index
      const float x = bf16_lo(w4[j]), y = bf16_hi(w4[j]);
      const float c = cs[i], sn = cs[32 + i];
      const float xr = x * c - y * sn, yr = x * sn + y * c;
      w4[j] = pack_bf16x2(xr, yr);
      lo4[j] = pack_bf16x2(xr - bf16_lo(w4[j]), yr - bf16_hi(w4[j]));
    }
    *q4 = make_uint4(w4[0], w4[1], w4[2], w4[3]);
    *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(q4) + NH * 128) = make_uint4(lo4[0], lo4[1], lo4[2], lo4[3]);
  }
}

// Reduces v[0..8) over the warp's 32 lanes: three halving exchange steps leave lane l with
// element (l >> 2) & 7 reduced over the 8 lanes that share bits 0..1 of l, two more steps
// complete it over all 32 lanes (result in v[0]; 9 shuffles).
template <bool MAX>
__device__ __forceinline__ void group_reduce8(float (&v)[8]) {
  const int ln = threadIdx.x & 31;
#pragma unroll
  for (int s = 0; s < 3; ++s) {
    const int half = 4 >> s, o = 16 >> s;
    const bool upper = (ln & o) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (i < half) {
        const float keep = upper ? v[i + half] : v[i];
        const float send = upper ? v[i] : v[i + half];
        const float got = __shfl_xor_sync(0xffffffffu, send, o);
        v[i] = MAX ? fmaxf(keep, got) : keep + got;
      }
    }
  }
#pragma unroll
  for (int o = 2; o >= 1; o >>= 1) {
    const float got = __shfl_xor_sync(0xffffffffu, v[0], o);
    v[0] = MAX ? fmaxf(v[0], got) : v[0] + got;
  }
}

// Four K-steps of 16 over one 64-dim panel of two K-major 128-byte-swizzled operands (32
// bytes apart); `acc` = accumulate into D from the first step on.
__device__ __forceinline__ void mma4(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, bool acc) {
  tc05::mma_bf16(d, ad, bd, idesc, acc ? 1u : 0u);
#pragma unroll
  for (int k = 1; k < 4; ++k) tc05::mma_bf16(d, tc05::desc_adv(ad, 32 * k), tc05::desc_adv(bd, 32 * k), idesc, 1u);
}
// S^T = K q'^T over the tile's eight 64-dim panels (16 KB apart) against the query's (QPANEL
// apart), then the low parts of the rotated query (ninth query panel) against the rotary panel.
template <int QPANEL>
__device__ __forceinline__ void gemm1_issue(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc) {
#pragma unroll 1
  for (int pnl = 0; pnl < 8; ++pnl)
    mma4(d, tc05::desc_adv(ad, pnl * kKPanel), tc05::desc_adv(bd, pnl * QPANEL), idesc, pnl > 0);
  mma4(d, tc05::desc_adv(ad, 7 * kKPanel), tc05::desc_adv(bd, 8 * QPANEL), idesc, true);
}
// One 128-dim chunk of O^T += V^T [P_hi | P_lo]^T: eight K-steps of 16 entries (2 KB apart in
// both MN-major operands); `acc` = accumulate into D from the first step on.
__device__ __forceinline__ void gemm2_chunk_issue(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, bool acc) {
  tc05::mma_bf16(d, ad, bd, idesc, acc ? 1u : 0u);
#pragma unroll
  for (int kk = 1; kk < kTileE / 16; ++kk)
    tc05::mma_bf16(d, tc05::desc_adv(ad, 2048 * kk), tc05::desc_adv(bd, 2048 * kk), idesc, 1u);
}

__device__ __forceinline__ void report_timeout_attn(int* flag, int32_t* dev_status) {
  atomicExch(flag, 1);
  if (dev_status != nullptr) atomicExch(dev_status, (int)CSA2_ETIMEOUT);
}

// One block: tile t (entries 128t .. 128t+127) of query row blockIdx.x, for NH of the 64
// heads (NH = 64, or 32 / 16 where rows x tiles alone would leave most SMs idle: the heads
// split across 64 / NH blocks, each gathering the tile).  Warp 0 allocates tensor memory and
// issues the MMAs (one thread); every warp gathers, runs the softmax for 32 entries x NH / 2
// heads (one thread per TMEM lane = entry) and writes partials.
template <int NH>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_tc05_kernel(const AttnParams p) {
  constexpr int HALF = NH / 2;            // heads of a warp's softmax share
  constexpr int NG = HALF / 8;            // groups of 8 of them
  constexpr int QPANEL = NH * 128;        // one 64-dim panel of the query: NH rows x 128 B
  constexpr int NO = 2 * NH;              // second GEMM's N: P_hi | P_lo
  constexpr uint32_t kCols = 4 * NO;      // tensor memory: O^T, four chunks of 128 dims
  constexpr int HS = kHeads / NH;         // blocks per tile
  static_assert(NH == 64 || NH == 32 || NH == 16, "heads per block");
  static_assert(9 * QPANEL <= kQBytes, "query panels fit");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1k(smem_raw);
  uint8_t* qs = smem;              // q' (first GEMM), then P_hi | P_lo (second GEMM)
  uint8_t* ks = smem + kQBytes;    // the latent tile
  AttnShared& sh = *reinterpret_cast<AttnShared*>(ks + kKBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // blockIdx.y = HS k + head group orders the tiles so that the window-only tiles (which need
  // nothing from the previous kernel) come first; tile = (k + tiles holding selected entries)
  // mod tiles
  const int row = blockIdx.x, n_tiles = gridDim.y / HS, h0 = (blockIdx.y % HS) * NH;
  const int sel_tiles = min(n_tiles, (p.K + kTileE - 1) / kTileE);
  const int tile = (blockIdx.y / HS + sel_tiles) % n_tiles;
  const bool needs_idx = tile * kTileE < p.K;
  const int b = p.seq_of_row[row];
  const long long qp = p.q_pos[row];
  const long long pos0 = p.swa_pos0[b];
  const long long lo = max(qp - (long long)p.window + 1, pos0);

  if (tid == 0) {
    tc05::mbar_init(&sh.bar_s, 1);
    tc05::mbar_init(&sh.bar_o, 1);
    sh.timeout = 0;
    sh.s_issued = sh.o_issued = 0;
    tc05::fence_barrier_init();
  }
  if (warp == 0) tc05::tmem_alloc(&sh.tmem_base, kCols);
  rope_table(sh.cs, p, qp, 1.f);
  // the next kernel in the stream may launch now (it waits for this grid before reading)
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  tc05::fence_before();
  __syncthreads();
  tc05::fence_after();
  const uint32_t tmem = sh.tmem_base;
  // one block per row hands its rotary table to the merge
  if (p.rope_cs != nullptr && blockIdx.y == 0 && tid < kRopeDim) p.rope_cs[(size_t)row * kRopeDim + tid] = sh.cs[tid];

  // the query is an input of the step, not of the previous kernel: it is copied and rotated
  // before the wait below
  copy_query<NH>(p, row, h0, qs);
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  rotate_query<NH>(qs, sh.cs);
  // With programmatic dependent launch this block may run while the kernel that writes the
  // selected indices is still finishing: tiles with selected entries wait for it here.
  if (needs_idx) asm volatile("griddepcontrol.wait;\n" ::: "memory");
  if (tid < kTileE) {
    const EntrySrc s = entry_source(p, row, b, qp, lo, pos0, tile * kTileE + tid);
    sh.src.ptr[tid] = s.valid ? s.ptr : nullptr;
    sh.src.sptr[tid] = s.sptr;
    sh.src.rs[tid] = s.rs;
    sh.src.fmt[tid] = s.valid ? s.fmt : -1;
  }
  __syncthreads();
  gather_tile(sh.src, ks, p.q);
  cp_async_commit();
  cp_async_wait<0>();
  // generic-proxy writes (cp.async and stores) become visible to the tensor cores
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  tc05::fence_before();
  __syncthreads();
  tc05::fence_after();

  const uint32_t qs_u = smem_u32(qs), ks_u = smem_u32(ks);
  // ---------------------------------------------------------------- S^T = K q'^T
  if (warp == 0) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc05::idesc_bf16(128, NH);
      const uint64_t ad = tc05::sw128_desc(ks_u), bd = tc05::sw128_desc(qs_u);
      gemm1_issue<QPANEL>(tmem, ad, bd, idesc);
      tc05::mma_commit(&sh.bar_s);
      sh.s_issued = 1;
    }
    __syncwarp();
  }

  // ---------------------------------------------------------------- softmax over the tile
  // warp w: TMEM lanes 32*(w&3) .. +31 (entry e = one lane), heads HALF*(w>>2) .. + HALF - 1
  // of the block's NH, in groups of 8 (rolled loops keep this run-once code small enough for
  // the instruction cache)
  const int qw = warp & 3, hb = HALF * (warp >> 2), e = 32 * qw + lane;
  const int lh = (lane >> 2) & 7;  // head within a group of 8 whose result this lane ends with
  {
    const bool ok = tc05::mbar_wait(&sh.bar_s, 0);
    if (!ok && lane == 0) report_timeout_attn(&sh.timeout, p.dev_status);
    tc05::fence_after();
    const int f = sh.src.fmt[e];
    const float rs = sh.src.rs[e];
    const bool on = ok && f >= 0;  // off: masked entry (logit -inf)
    const float zs = p.scale * rs;
    const uint32_t trow = tmem + ((uint32_t)(32 * qw) << 16) + (uint32_t)hb;
    // the thread's HALF logits (entry e, heads hb .. hb + HALF - 1) stay in registers for both
    // passes
    float z[HALF];
    {
      uint32_t v[HALF];
      tc05::tmem_ld<HALF>(trow, v);
      tc05::tmem_ld_wait();
#pragma unroll
      for (int k = 0; k < HALF; ++k) z[k] = on ? __uint_as_float(v[k]) * zs : -INFINITY;
    }
    // per-head maximum over the tile's entries
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      float m[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) m[k] = z[8 * g + k];
      group_reduce8<true>(m);
      if ((lane & 3) == 0) sh.red[qw][hb + 8 * g + lh] = m[0];
    }
    __syncthreads();
    if (qw == 0 && lane < HALF)
      sh.mfin[hb + lane] = fmaxf(fmaxf(sh.red[0][hb + lane], sh.red[1][hb + lane]),
                                 fmaxf(sh.red[2][hb + lane], sh.red[3][hb + lane]));
    __syncthreads();
    // P = exp(z - M) as P_hi | P_lo rows (entry e, MN-major for the second GEMM: 64 heads of
    // P_hi in one 128-byte row and P_lo in a second chunk kPBytes on; with fewer heads P_lo
    // follows P_hi in the same row), the FP8 row scale on the weights; per-head sums of the
    // unscaled P
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const float4 m0 = *reinterpret_cast<const float4*>(&sh.mfin[hb + 8 * g]);
      const float4 m1 = *reinterpret_cast<const float4*>(&sh.mfin[hb + 8 * g + 4]);
      const float M[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
      float pe[8];
      uint32_t hi[4], lw[4];
#pragma unroll
      for (int k = 0; k < 8; ++k) pe[k] = on ? __expf(z[8 * g + k] - (M[k] == -INFINITY ? 0.f : M[k])) : 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float a0 = pe[2 * k] * rs, a1 = pe[2 * k + 1] * rs;
        hi[k] = pack_bf16x2(a0, a1);
        lw[k] = pack_bf16x2(a0 - bf16_lo(hi[k]), a1 - bf16_hi(hi[k]));
      }
      const int ci = hb / 8 + g;  // 16-byte chunk of this group's heads
      const int off = e * 128 + ((ci ^ (e & 7)) << 4);
      const int off_lo = NH == 64 ? kPBytes + off : e * 128 + (((NH / 8 + ci) ^ (e & 7)) << 4);
      *reinterpret_cast<uint4*>(qs + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(qs + off_lo) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      group_reduce8<false>(pe);
      if ((lane & 3) == 0) sh.red_sum[qw][hb + 8 * g + lh] = pe[0];
    }
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  }
  tc05::fence_before();
  __syncthreads();
  tc05::fence_after();

  // ---------------------------------------------------------------- O^T = V^T [P_hi | P_lo]^T
  // S^T is dead now: chunk c of 128 dims accumulates into columns NO*c .. NO*c + NO - 1, the
  // P_hi products in the first NH, the P_lo products in the last NH.
  if (warp == 0) {
    if (lane == 0 && !sh.timeout) {
      // A = V^T (dims x entries, MN-major: 64-dim panels 16 KB apart, 8-entry groups 1 KB
      // apart); B = [P_hi | P_lo]^T (entries x 128, MN-major: two 64-column chunks 16 KB
      // apart, 8-entry groups 1 KB apart)
      constexpr uint32_t idesc = tc05::idesc_bf16(128, NO) | (1u << 15) | (1u << 16);
#pragma unroll 1
      for (int c = 0; c < 4; ++c)
        gemm2_chunk_issue(tmem + NO * c, sw128_desc_lbo(ks_u + 2 * c * kKPanel, kKPanel, 1024),
                          sw128_desc_lbo(qs_u, kPBytes, 1024), idesc, false);
      tc05::mma_commit(&sh.bar_o);
      sh.o_issued = 1;
    }
    __syncwarp();
  }
  __syncthreads();

  // ---------------------------------------------------------------- partial results
  // part_o[row][tile][h][d] = O[h][d] (relative to M_h); warp w reads TMEM lanes 32*(w&3) of
  // dim chunks 2*(w>>2), 2*(w>>2)+1: thread -> one dim, 8 heads per step
  const bool live = sh.o_issued && tc05::mbar_wait(&sh.bar_o, 0);
  if (!live && sh.o_issued && lane == 0) report_timeout_attn(&sh.timeout, p.dev_status);
  tc05::fence_after();
  if (live) {
    constexpr int W = NH < 32 ? NH : 32;  // heads per TMEM load
    float* po = p.part_o + (((size_t)row * n_tiles + tile) * kHeads + h0) * kHeadDim;
#pragma unroll 1
    for (int i = 0; i < 2 * (NH / W); ++i) {
      const int c = 2 * (warp >> 2) + i / (NH / W), g = i % (NH / W);  // heads W*g .. of dim chunk c
      const int d = 128 * c + 32 * qw + lane;
      uint32_t vh[W], vl[W];
      const uint32_t ta = tmem + ((uint32_t)(32 * qw) << 16) + NO * c + W * g;
      tc05::tmem_ld<W>(ta, vh);
      tc05::tmem_ld<W>(ta + NH, vl);
      tc05::tmem_ld_wait();
#pragma unroll
      for (int k = 0; k < W; ++k)
        po[(size_t)(W * g + k) * kHeadDim + d] = __uint_as_float(vh[k]) + __uint_as_float(vl[k]);
    }
  }
  if (warp == 4) {
    float* pm = p.part_ml + (((size_t)row * n_tiles + tile) * kHeads + h0) * 2;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int h = 2 * lane + j;
      if (h < NH) {
        const float l = (sh.red_sum[0][h] + sh.red_sum[1][h]) + (sh.red_sum[2][h] + sh.red_sum[3][h]);
        pm[2 * h] = live ? sh.mfin[h] : -INFINITY;
        pm[2 * h + 1] = live ? l : 0.f;
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc05::fence_before();
  __syncthreads();
  if (sh.timeout && tid == 0) {
    // let issued MMAs finish (bounded) before the tensor memory is freed
    if (sh.s_issued) tc05::mbar_wait(&sh.bar_s, 0);
    if (sh.o_issued) tc05::mbar_wait(&sh.bar_o, 0);
  }
  __syncthreads();
  if (warp == 0) {
    tc05::fence_after();
    tc05::tmem_dealloc(tmem, kCols);
  }
}

// ===================================================================================== rows
// One block: every tile of query row blockIdx.x for the NH heads h0 = NH * blockIdx.y .., one
// tile after another with the softmax carried across the tiles.  Each head keeps a reference
// maximum M: the first tile's maximum, moved only when a later tile's maximum exceeds it by
// more than kRowTau (the output accumulated in tensor memory and the running sum are then
// scaled by exp(M_old - M_new)), so P = exp(z - M) <= e^kRowTau and every tile's second GEMM
// accumulates into the same tensor memory.  After the last tile the sink joins the
// denominator, the output is normalised, its rotary coordinates are turned back by -position
// and it is written directly: no partials and no merge kernel.  The window tile (which needs
// nothing from the previous kernel) comes first.
constexpr float kRowTau = 8.f;

struct RowShared {
  TileSrc src;
  float red[4][32];  // per TMEM lane quarter: per-head maxima, then sums, over its 32 entries
  float mref[32];    // reference maximum per head
  float alpha[32];   // this tile's rescale factor per head (1: unchanged), then the output factor
  float lsum[32];    // running sum of P per head, relative to mref
  float cs[kRopeDim];
  uint64_t bar_s, bar_o;  // first / second GEMM of the current tile completed
  uint32_t tmem_base;
  int timeout;
  int rescale;  // some head's reference moved at this tile
  int s_issued, o_issued;  // tiles whose first / second GEMM was issued
};

template <int NH>
constexpr int row_smem_bytes() {
  return 1024 + 9 * NH * 128 + kPBytes + kKBytes + (int)sizeof(RowShared);
}

template <int NH>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_row_kernel(const AttnParams p) {
  constexpr int HALF = NH / 2;            // heads of a warp's softmax share
  constexpr int NG = HALF / 8;            // groups of 8 of them
  constexpr int QPANEL = NH * 128;        // one 64-dim panel of the query
  constexpr int NO = 2 * NH;              // second GEMM's N: P_hi | P_lo
  constexpr uint32_t kS0 = 4 * NO;        // tensor memory: O in [0, kS0), S^T in [kS0, kS0 + NH)
  constexpr uint32_t kCols = NH == 32 ? 512 : 256;
  static_assert(NH == 16 || NH == 32, "heads per block");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1k(smem_raw);
  uint8_t* qs = smem;                     // q' (nine panels), kept for every tile
  uint8_t* ps = qs + 9 * QPANEL;          // P_hi | P_lo of the current tile
  uint8_t* ks = ps + kPBytes;             // the current tile's latents
  RowShared& sh = *reinterpret_cast<RowShared*>(ks + kKBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = blockIdx.x, h0 = blockIdx.y * NH;
  const int n_tiles = (p.K + p.window + kTileE - 1) / kTileE;
  const int sel_tiles = min(n_tiles, (p.K + kTileE - 1) / kTileE);
  const int b = p.seq_of_row[row];
  const long long qp = p.q_pos[row];
  const long long pos0 = p.swa_pos0[b];
  const long long lo = max(qp - (long long)p.window + 1, pos0);

  if (tid == 0) {
    tc05::mbar_init(&sh.bar_s, 1);
    tc05::mbar_init(&sh.bar_o, 1);
    sh.timeout = 0;
    sh.rescale = 0;
    sh.s_issued = sh.o_issued = 0;
    tc05::fence_barrier_init();
  }
  if (warp == 0) tc05::tmem_alloc(&sh.tmem_base, kCols);
  rope_table(sh.cs, p, qp, 1.f);
  if (tid < NH) {
    sh.mref[tid] = -INFINITY;
    sh.lsum[tid] = 0.f;
  }
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  tc05::fence_before();
  __syncthreads();
  tc05::fence_after();
  const uint32_t tmem = sh.tmem_base;
  const uint32_t qs_u = smem_u32(qs), ps_u = smem_u32(ps), ks_u = smem_u32(ks);

  // the query is an input of the step: copied and rotated before any wait
  copy_query<NH>(p, row, h0, qs);
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  rotate_query<NH>(qs, sh.cs);

  const int qw = warp & 3, hb = HALF * (warp >> 2), e = 32 * qw + lane;
  const int lh = (lane >> 2) & 7;  // head within a group of 8 whose result this lane ends with
  bool waited = false;
#pragma unroll 1
  for (int kt = 0; kt < n_tiles; ++kt) {
    const int tile = (kt + sel_tiles) % n_tiles;
    // tiles with selected entries wait for the kernel that writes the indices
    if (!waited && tile * kTileE < p.K) {
      asm volatile("griddepcontrol.wait;\n" ::: "memory");
      waited = true;
    }
    // the previous tile's second GEMM is done: its latents and P may be overwritten
    if (kt > 0 && !sh.timeout && !tc05::mbar_wait(&sh.bar_o, (kt - 1) & 1) && lane == 0)
      report_timeout_attn(&sh.timeout, p.dev_status);
    if (tid < kTileE) {
      const EntrySrc sr = entry_source(p, row, b, qp, lo, pos0, tile * kTileE + tid);
      sh.src.ptr[tid] = sr.valid ? sr.ptr : nullptr;
      sh.src.sptr[tid] = sr.sptr;
      sh.src.rs[tid] = sr.rs;
      sh.src.fmt[tid] = sr.valid ? sr.fmt : -1;
    }
    if (tid == 0) sh.rescale = 0;
    __syncthreads();
    gather_tile(sh.src, ks, p.q);
    cp_async_commit();
    cp_async_wait<0>();
    // generic-proxy writes (cp.async, stores, the rotated query) become visible to the tensor cores
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    tc05::fence_before();
    __syncthreads();
    tc05::fence_after();

    // ------------------------------------------------------------ S^T = K q'^T
    if (warp == 0) {
      if (lane == 0 && !sh.timeout) {
        constexpr uint32_t idesc = tc05::idesc_bf16(128, NH);
        gemm1_issue<QPANEL>(tmem + kS0, tc05::sw128_desc(ks_u), tc05::sw128_desc(qs_u), idesc);
        tc05::mma_commit(&sh.bar_s);
        sh.s_issued = kt + 1;
      }
      __syncwarp();
    }

    // ------------------------------------------------------------ softmax of the tile
    const bool ok = !sh.timeout && tc05::mbar_wait(&sh.bar_s, kt & 1);
    if (!ok && lane == 0 && !sh.timeout) report_timeout_attn(&sh.timeout, p.dev_status);
    tc05::fence_after();
    const int f = sh.src.fmt[e];
    const float rs = sh.src.rs[e];
    const bool on = ok && f >= 0;
    const float zs = p.scale * rs;
    float z[HALF];
    {
      uint32_t v[HALF];
      tc05::tmem_ld<HALF>(tmem + ((uint32_t)(32 * qw) << 16) + kS0 + (uint32_t)hb, v);
      tc05::tmem_ld_wait();
#pragma unroll
      for (int k = 0; k < HALF; ++k) z[k] = on ? __uint_as_float(v[k]) * zs : -INFINITY;
    }
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      float m[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) m[k] = z[8 * g + k];
      group_reduce8<true>(m);
      if ((lane & 3) == 0) sh.red[qw][hb + 8 * g + lh] = m[0];
    }
    __syncthreads();
    if (qw == 0 && lane < HALF) {
      // this tile's maximum; the reference moves when it is exceeded by more than kRowTau
      const int h = hb + lane;
      const float mt = fmaxf(fmaxf(sh.red[0][h], sh.red[1][h]), fmaxf(sh.red[2][h], sh.red[3][h]));
      const float mr = sh.mref[h];
      float a = 1.f;
      if (mr == -INFINITY) {
        sh.mref[h] = mt;  // first finite maximum: the accumulated output and sum are still zero
      } else if (mt > mr + kRowTau) {
        a = __expf(mr - mt);
        sh.mref[h] = mt;
        sh.rescale = 1;
      }
      sh.alpha[h] = a;
    }
    tc05::fence_before();
    __syncthreads();
    tc05::fence_after();
    if (sh.rescale && kt > 0) {
      // O *= alpha per head: lane l of TMEM holds dim 32 qw + l of each 128-dim chunk; columns
      // NO c + j are head j % NH (P_hi products, then P_lo products)
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * (warp >> 2) + cc;
#pragma unroll 1
        for (int part = 0; part < NO / 32; ++part) {
          const uint32_t ta = tmem + ((uint32_t)(32 * qw) << 16) + NO * c + 32 * part;
          uint32_t v[32];
          tc05::tmem_ld32(ta, v);
          tc05::tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * sh.alpha[(32 * part + k) % NH]);
          tc05::tmem_st32(ta, v);
        }
      }
      tc05::tmem_st_wait();
    }
    // P = exp(z - M) as P_hi | P_lo rows (entry e, MN-major for the second GEMM: P_hi in
    // columns 0 .. NH-1, P_lo in NH .. 2NH-1 of a 128-byte row), the FP8 row scale on the
    // weights; per-head sums of the unscaled P
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      float pe[8];
      uint32_t hi[4], lw[4];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float M = sh.mref[hb + 8 * g + k];
        pe[k] = on ? __expf(z[8 * g + k] - (M == -INFINITY ? 0.f : M)) : 0.f;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float a0 = pe[2 * k] * rs, a1 = pe[2 * k + 1] * rs;
        hi[k] = pack_bf16x2(a0, a1);
        lw[k] = pack_bf16x2(a0 - bf16_lo(hi[k]), a1 - bf16_hi(hi[k]));
      }
      const int ci = hb / 8 + g;
      *reinterpret_cast<uint4*>(ps + e * 128 + ((ci ^ (e & 7)) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(ps + e * 128 + (((NH / 8 + ci) ^ (e & 7)) << 4)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      group_reduce8<false>(pe);
      if ((lane & 3) == 0) sh.red[qw][hb + 8 * g + lh] = pe[0];
    }
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    tc05::fence_before();
    __syncthreads();
    tc05::fence_after();
    if (qw == 0 && lane < HALF) {
      const int h = hb + lane;
      sh.lsum[h] = sh.lsum[h] * sh.alpha[h] + ((sh.red[0][h] + sh.red[1][h]) + (sh.red[2][h] + sh.red[3][h]));
    }

    // ------------------------------------------------------------ O^T += V^T [P_hi | P_lo]^T
    if (warp == 0) {
      if (lane == 0 && !sh.timeout) {
        constexpr uint32_t idesc = tc05::idesc_bf16(128, NO) | (1u << 15) | (1u << 16);
#pragma unroll 1
        for (int c = 0; c < 4; ++c)
          gemm2_chunk_issue(tmem + NO * c, sw128_desc_lbo(ks_u + 2 * c * kKPanel, kKPanel, 1024),
                            sw128_desc_lbo(ps_u, kPBytes, 1024), idesc, kt > 0);
        tc05::mma_commit(&sh.bar_o);
        sh.o_issued = kt + 1;
      }
      __syncwarp();
    }
  }

  // ---------------------------------------------------------------- output
  __syncthreads();  // the last tile's running sums are final
  const bool live = !sh.timeout && tc05::mbar_wait(&sh.bar_o, (n_tiles - 1) & 1);
  if (!live && !sh.timeout && lane == 0) report_timeout_attn(&sh.timeout, p.dev_status);
  tc05::fence_after();
  if (tid < NH) {
    // the sink joins the denominator: o = O e^{M - Mf} / (l e^{M - Mf} + e^{sink - Mf})
    const float M = sh.mref[tid], sk = __ldg(p.sink + h0 + tid);
    const float Mf = fmaxf(M, sk);
    const float so = M == -INFINITY ? 0.f : __expf(M - Mf);
    const float es = __expf(sk - Mf);
    const float den = sh.lsum[tid] * so + es;
    sh.alpha[tid] = so / den;
    if (p.sink_mass) p.sink_mass[(size_t)row * kHeads + h0 + tid] = es / den;
  }
  __syncthreads();
  if (live) {
#pragma unroll 1
    for (int cc = 0; cc < 2; ++cc) {
      const int c = 2 * (warp >> 2) + cc;
      const int d = 128 * c + 32 * qw + lane;
      uint32_t v[32], v2[32];
      const uint32_t ta = tmem + ((uint32_t)(32 * qw) << 16) + NO * c;
      tc05::tmem_ld32(ta, v);
      if (NH == 32) tc05::tmem_ld32(ta + 32, v2);
      tc05::tmem_ld_wait();
      float o[NH];
#pragma unroll
      for (int k = 0; k < NH; ++k)
        o[k] = (NH == 32 ? __uint_as_float(v[k]) + __uint_as_float(v2[k])
                         : __uint_as_float(v[k]) + __uint_as_float(v[k + NH])) * sh.alpha[k];
      if (d >= kHeadDim - kRopeDim) {
        // turned back by -position: pairs (448 + 2i, 449 + 2i) sit in adjacent lanes
        const int i = (d - (kHeadDim - kRopeDim)) >> 1;
        const float cn = sh.cs[i], sn = sh.cs[32 + i];
        const bool even = (d & 1) == 0;
#pragma unroll
        for (int k = 0; k < NH; ++k) {
          const float other = __shfl_xor_sync(0xffffffffu, o[k], 1);
          o[k] = even ? o[k] * cn + other * sn : o[k] * cn - other * sn;
        }
      }
      const size_t at = ((size_t)row * kHeads + h0) * kHeadDim + d;
#pragma unroll
      for (int k = 0; k < NH; ++k) {
        if (p.out_bf16) static_cast<__nv_bfloat16*>(p.out)[at + (size_t)k * kHeadDim] = __float2bfloat16_rn(o[k]);
        else static_cast<float*>(p.out)[at + (size_t)k * kHeadDim] = o[k];
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc05::fence_before();
  __syncthreads();
  if (sh.timeout && tid == 0) {
    // let issued MMAs finish (bounded) before the tensor memory is freed
    if (sh.s_issued > 0) tc05::mbar_wait(&sh.bar_s, (sh.s_issued - 1) & 1);
    if (sh.o_issued > 0) tc05::mbar_wait(&sh.bar_o, (sh.o_issued - 1) & 1);
  }
  __syncthreads();
  if (warp == 0) {
    tc05::fence_after();
    tc05::tmem_dealloc(tmem, kCols);
  }
}

// ===================================================================================== pipeline
// Batches of many rows (a prefill chunk: thousands of query rows): one block per (row, 32
// heads) over all of the row's tiles, as in the row kernel, with the tile stream pipelined
// across warp roles so that a tile's copies overlap the previous tile's arithmetic:
//   copies             the latent rows go by cp.async into a ring of five 32 KB slots, one
//                      slot per pair of 64-dim panels (fill u = pair u mod 4 of tile u / 4
//                      goes to slot u mod 5); the copy warps (4) form each tile's entry
//                      sources and copy its pairs 0 and 1, the two halves of the softmax
//                      warps copy pairs 2 and 3 before the tile's softmax (they would
//                      otherwise wait for it idle); each group of 128 threads reports its slot
//                      full once its copies have landed;
//   MMA thread         S^T = K q'^T pair by pair as the slots fill; then, once the softmax has
//                      written P, O^T += V^T [P_hi | P_lo]^T chunk by chunk, each chunk's
//                      commit freeing the slot it read;
//   softmax warps (8)  as in the row kernel: a reference maximum per head that moves only by
//                      more than kRowTau (the output in tensor memory rescaled then), P to
//                      shared memory as hi + lo bf16 terms, running sums.
// Tile t+1's first pair goes to the fifth slot while tile t is processed, its other pairs as
// tile t's second GEMM frees slots.  MMAs complete in issue order, so once the softmax sees
// tile t+1's logits, tile t's second GEMM has finished: P (one buffer) may be rewritten and
// the output rescaled.  bf16 latents and window rows only (they are copied as they are).
constexpr int kPipeThreads = 512;     // warp 0 MMA, warps 4..11 softmax, warps 12..15 copies
constexpr int kPipeSoftFirst = 4, kPipeCopyFirst = 12;
constexpr int kPipeSlots = 5;
constexpr int kPipeSlotBytes = 2 * kKPanel;  // 32 KB: 128 entries x 128 dims
constexpr int kPipeNH = 32;
constexpr uint32_t kPipeSpin = 1u << 20;

struct PipeShared {
  const uint8_t* ptr[2][kTileE];  // per tile parity: entry rows
  int fmt[2][kTileE];          // per tile parity: entry format, -1 = masked
  float rs[2][kTileE];         // per tile parity: FP8 row scale (1 for bf16)
  float red_max[4][32];        // per TMEM lane quarter: per-head maxima over its 32 entries
  float red_sum[4][32];        // ... and sums of P
  float mref[32], alpha[32], lsum[32];
  float cs[kRopeDim];
  uint64_t full[kPipeSlots], empty[kPipeSlots];  // slot filled (copies) / freed (second GEMM)
  uint64_t src_ready[2];                          // per tile parity: the entry sources are written
  uint64_t s_full, p_full, o_done, fin;           // first GEMM done / P written / last GEMM / all MMAs
  uint32_t tmem_base;
  int timeout;
  int rescale_tile;  // last tile at which some head's reference moved
};

constexpr int pipe_smem_bytes() {
  return 1024 + 9 * kPipeNH * 128 + kPBytes + kPipeSlots * kPipeSlotBytes + (int)sizeof(PipeShared);
}
static_assert(pipe_smem_bytes() <= 232448, "the pipeline's shared memory fits one block per SM");

// Bounded wait that also gives up when another role has recorded a timeout.
__device__ __forceinline__ bool pipe_wait(uint64_t* bar, uint32_t parity, const int* abort) {
  const uint32_t a = smem_u32(bar);
  for (uint32_t i = 0; i < kPipeSpin; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred P1;\n mbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2;\n selp.b32 %0, 1, 0, P1;\n}\n"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
    if (*reinterpret_cast<const volatile int*>(abort)) return false;
  }
  return false;
}

// Barrier `id` over `count` threads (whole warps, converged first).
__device__ __forceinline__ void named_bar(int id, int count) {
  __syncwarp();
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}

// Pair c of tile t (fill u = 4t + c) by 128 threads (thread g: 16-byte chunk g & 15 of the
// pair's 256 bytes of entries (g >> 4) + 8k): waits for the slot, copies, and reports the slot
// full once its copies have landed.  Returns false after a failed wait (warp-uniform).
__device__ __forceinline__ bool pipe_copy_pair(PipeShared& sh, uint8_t* ring, int t, int c, int g, int32_t* dev_status) {
  const int u = 4 * t + c, slot = u % kPipeSlots;
  const bool got = pipe_wait(&sh.empty[slot], ((u / kPipeSlots) & 1) ^ 1, &sh.timeout);
  if (!__all_sync(0xffffffffu, got)) {
    if (!sh.timeout) report_timeout_attn(&sh.timeout, dev_status);
    return false;
  }
  uint8_t* dst = ring + slot * kPipeSlotBytes;
  const int j = g & 15, r0 = g >> 4;
  const uint8_t* const* ptr = sh.ptr[t & 1];
  const int* fmt = sh.fmt[t & 1];
#pragma unroll 4
  for (int k = 0; k < kTileE / 8; ++k) {
    const int r = r0 + 8 * k;
    cp_async16(dst + sw128_off(r, j, kTileE), ptr[r] + 256 * c + 16 * j, fmt[r] >= 0);
  }
  cp_async_commit();
  cp_async_wait<0>();
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // the copies are read by the tensor cores
  tc05::mbar_arrive(&sh.full[slot]);
  return true;
}

__global__ void __launch_bounds__(kPipeThreads, 1) attn_pipe_kernel(const AttnParams p) {
  constexpr int NH = kPipeNH, HALF = NH / 2, NG = HALF / 8;
  constexpr int QPANEL = NH * 128;
  constexpr int NO = 2 * NH;              // second GEMM's N: P_hi | P_lo
  constexpr uint32_t kS0 = 4 * NO;        // tensor memory: O in [0, kS0), two S^T buffers from kS0
  constexpr uint32_t kCols = 512;
  static_assert(kS0 + 2 * NH <= kCols, "output and two logit buffers fit");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1k(smem_raw);
  uint8_t* qs = smem;                     // q' (nine panels), kept for every tile
  uint8_t* ps = qs + 9 * QPANEL;          // P_hi | P_lo of the current tile
  uint8_t* ring = ps + kPBytes;           // five slots of two latent panels
  PipeShared& sh = *reinterpret_cast<PipeShared*>(ring + kPipeSlots * kPipeSlotBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = blockIdx.x, h0 = blockIdx.y * NH;
  const int n_tiles = (p.K + p.window + kTileE - 1) / kTileE;
  const int sel_tiles = min(n_tiles, (p.K + kTileE - 1) / kTileE);
  const int b = p.seq_of_row[row];
  const long long qp = p.q_pos[row];
  const long long pos0 = p.swa_pos0[b];
  const long long lo = max(qp - (long long)p.window + 1, pos0);

  if (tid == 0) {
    for (int i = 0; i < kPipeSlots; ++i) {
      tc05::mbar_init(&sh.full[i], kTileE);  // one arrive per copy thread
      tc05::mbar_init(&sh.empty[i], 1);
    }
    tc05::mbar_init(&sh.s_full, 1);
    tc05::mbar_init(&sh.p_full, 1);
    tc05::mbar_init(&sh.o_done, 1);
    tc05::mbar_init(&sh.fin, 1);
    tc05::mbar_init(&sh.src_ready[0], 1);
    tc05::mbar_init(&sh.src_ready[1], 1);
    sh.timeout = 0;
    sh.rescale_tile = -1;
    tc05::fence_barrier_init();
  }
  if (warp == 0) tc05::tmem_alloc(&sh.tmem_base, kCols);
  rope_table(sh.cs, p, qp, 1.f);
  if (tid < NH) {
    sh.mref[tid] = -INFINITY;
    sh.lsum[tid] = 0.f;
  }
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  __syncthreads();
  // the query is an input of the step: copied and rotated before any wait
  if (tid < kAttnThreads) copy_query<NH>(p, row, h0, qs);
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  if (tid < kAttnThreads) rotate_query<NH>(qs, sh.cs);
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // q' is read by the tensor cores
  tc05::fence_before();
  __syncthreads();
  tc05::fence_after();
  const uint32_t tmem = sh.tmem_base;
  const uint32_t qs_u = smem_u32(qs), ps_u = smem_u32(ps), ring_u = smem_u32(ring);

  if (warp >= kPipeCopyFirst) {
    // ---------------------------------------------------------------- copies: sources, pairs 0 and 1
    const int g = tid - kPipeCopyFirst * 32;  // entry g of each tile
    bool waited = false, ok = true;
    // every copy thread runs every iteration (the named barriers); after a failed wait it only
    // skips the work
#pragma unroll 1
    for (int t = 0; t < n_tiles; ++t) {
      const int tile = (t + sel_tiles) % n_tiles;
      if (!waited && tile * kTileE < p.K) {  // the selected indices come from the previous kernel
        asm volatile("griddepcontrol.wait;\n" ::: "memory");
        waited = true;
      }
      // parity t & 1 was last read for tile t - 2, whose softmax (and so its copies) finished
      // before the slot this loop waited on for tile t - 1's pair 1 was freed
      const EntrySrc sr = entry_source(p, row, b, qp, lo, pos0, tile * kTileE + g);
      sh.ptr[t & 1][g] = sr.valid ? sr.ptr : reinterpret_cast<const uint8_t*>(p.q);
      sh.fmt[t & 1][g] = sr.valid ? sr.fmt : -1;
      sh.rs[t & 1][g] = sr.rs;
      named_bar(2, 128);
      if (g == 0) tc05::mbar_arrive(&sh.src_ready[t & 1]);
      if (ok) {
        ok = pipe_copy_pair(sh, ring, t, 0, g, p.dev_status) && pipe_copy_pair(sh, ring, t, 1, g, p.dev_status);
      }
    }
    cp_async_wait<0>();
  } else if (warp == 0) {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      bool ok = true;
      constexpr uint32_t idesc1 = tc05::idesc_bf16(128, NH);
      constexpr uint32_t idesc2 = tc05::idesc_bf16(128, NO) | (1u << 15) | (1u << 16);
      const uint64_t qd = tc05::sw128_desc(qs_u), pd = sw128_desc_lbo(ps_u, kPBytes, 1024);
      // S^T(t) = K q'^T, pair c, into logit buffer t & 1 (the caller made sure the pair landed)
      auto gemm1_pair = [&](int t, int c) {
        const int slot = (4 * t + c) % kPipeSlots;
        const uint32_t sc = tmem + kS0 + (uint32_t)(t & 1) * NH;
        const uint64_t ad = tc05::sw128_desc(ring_u + slot * kPipeSlotBytes);
        const uint64_t bd = tc05::desc_adv(qd, 2 * c * QPANEL);
        mma4(sc, ad, bd, idesc1, c > 0);
        mma4(sc, tc05::desc_adv(ad, kKPanel), tc05::desc_adv(bd, QPANEL), idesc1, true);
        // the low parts of the rotated query against the rotary panel (the last pair's second)
        if (c == 3) mma4(sc, tc05::desc_adv(ad, kKPanel), tc05::desc_adv(qd, 8 * QPANEL), idesc1, true);
      };
      auto wait_pair = [&](int t, int c) {
        const int u = 4 * t + c;
        if (!pipe_wait(&sh.full[u % kPipeSlots], (u / kPipeSlots) & 1, &sh.timeout)) return false;
        tc05::fence_after();
        return true;
      };
      // tile 0's first GEMM
#pragma unroll 1
      for (int c = 0; c < 4 && ok; ++c) {
        ok = wait_pair(0, c);
        if (ok) gemm1_pair(0, c);
      }
      if (ok) tc05::mma_commit(&sh.s_full);
#pragma unroll 1
      for (int t = 0; t < n_tiles && ok; ++t) {
        // the next tile's first pair (the spare slot) goes in while this tile's softmax runs,
        // if it has landed (its own logit buffer: the softmax reads buffer t & 1)
        int next_c = 0;
        if (t + 1 < n_tiles) {
          const int u = 4 * (t + 1);
          if (tc05::mbar_test(&sh.full[u % kPipeSlots], (u / kPipeSlots) & 1)) {
            tc05::fence_after();
            gemm1_pair(t + 1, 0);
            next_c = 1;
          }
        }
        // O^T += V^T [P_hi | P_lo]^T once the softmax has written P
        if (!pipe_wait(&sh.p_full, t & 1, &sh.timeout)) {
          ok = false;
          break;
        }
        tc05::fence_after();
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          const int slot = (4 * t + c) % kPipeSlots;
          gemm2_chunk_issue(tmem + NO * c, sw128_desc_lbo(ring_u + slot * kPipeSlotBytes, kKPanel, 1024), pd, idesc2,
                            t > 0);
          tc05::mma_commit(&sh.empty[slot]);
        }
        // the rest of the next tile's first GEMM as its pairs land (the slots this GEMM freed)
        if (t + 1 < n_tiles) {
#pragma unroll 1
          for (int c = next_c; c < 4 && ok; ++c) {
            ok = wait_pair(t + 1, c);
            if (ok) gemm1_pair(t + 1, c);
          }
          // its commit also covers this tile's second GEMM: the softmax of tile t + 1 may
          // rescale the output and rewrite P once it sees the logits
          if (ok) tc05::mma_commit(&sh.s_full);
        }
      }
      if (ok) tc05::mma_commit(&sh.o_done);
      else if (!sh.timeout) report_timeout_attn(&sh.timeout, p.dev_status);
      // every MMA issued has completed before the tensor memory is freed
      tc05::mma_commit(&sh.fin);
      tc05::mbar_wait(&sh.fin, 0);
    }
    __syncwarp();
  } else if (warp >= kPipeSoftFirst) {
    // ---------------------------------------------------------------- softmax
    const int sw = warp - kPipeSoftFirst;
    const int qw = sw & 3, hb = HALF * (sw >> 2), e = 32 * qw + lane;
    const int lh = (lane >> 2) & 7;  // head within a group of 8 whose result this lane ends with
    const uint32_t lane_base = tmem + ((uint32_t)(32 * qw) << 16);
    const int cgrp = sw >> 2, cg = tid - (kPipeSoftFirst + 4 * cgrp) * 32;  // copies pair 2 + cgrp
    bool ok = true;
    // every softmax thread runs every iteration (the named barriers); after a failed wait it
    // computes nothing that reaches tensor memory or the MMA thread
#pragma unroll 1
    for (int t = 0; t < n_tiles; ++t) {
      // this half's pair of the tile, once the copy warps have written its sources
      if (ok) {
        const bool src = pipe_wait(&sh.src_ready[t & 1], (t >> 1) & 1, &sh.timeout);
        ok = __all_sync(0xffffffffu, src) && pipe_copy_pair(sh, ring, t, 2 + cgrp, cg, p.dev_status);
        if (!ok && !sh.timeout) report_timeout_attn(&sh.timeout, p.dev_status);
      }
      // warp-uniform: the tensor-memory loads and stores below are warp-wide
      ok = __all_sync(0xffffffffu, ok && pipe_wait(&sh.s_full, t & 1, &sh.timeout));
      tc05::fence_after();
      const int f = sh.fmt[t & 1][e];
      const float rs = sh.rs[t & 1][e];
      const bool on = ok && f >= 0;
      const float zs = p.scale * rs;
      float z[HALF];
      if (ok) {
        uint32_t v[HALF];
        tc05::tmem_ld<HALF>(lane_base + kS0 + (uint32_t)(t & 1) * NH + (uint32_t)hb, v);
        tc05::tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < HALF; ++k) z[k] = on ? __uint_as_float(v[k]) * zs : -INFINITY;
      } else {
#pragma unroll
        for (int k = 0; k < HALF; ++k) z[k] = -INFINITY;
      }
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) {
        float m[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) m[k] = z[8 * gi + k];
        group_reduce8<true>(m);
        if ((lane & 3) == 0) sh.red_max[qw][hb + 8 * gi + lh] = m[0];
      }
      named_bar(1, 256);
      if (qw == 0 && lane < HALF) {
        const int h = hb + lane;
        const float mt = fmaxf(fmaxf(sh.red_max[0][h], sh.red_max[1][h]), fmaxf(sh.red_max[2][h], sh.red_max[3][h]));
        const float mr = sh.mref[h];
        float a = 1.f;
        if (mr == -INFINITY) {
          sh.mref[h] = mt;  // first finite maximum: the accumulated output and sum are still zero
        } else if (mt > mr + kRowTau) {
          a = __expf(mr - mt);
          sh.mref[h] = mt;
          sh.rescale_tile = t;
        }
        sh.alpha[h] = a;
      }
      named_bar(1, 256);
      if (ok && sh.rescale_tile == t && t > 0) {
        // O *= alpha per head (the previous tile's second GEMM has completed: this tile's
        // first GEMM was issued after it and has completed)
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * (sw >> 2) + cc;
#pragma unroll 1
          for (int part = 0; part < NO / 32; ++part) {
            const uint32_t ta = lane_base + NO * c + 32 * part;
            uint32_t v[32];
            tc05::tmem_ld32(ta, v);
            tc05::tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * sh.alpha[(32 * part + k) % NH]);
            tc05::tmem_st32(ta, v);
          }
        }
        tc05::tmem_st_wait();
      }
      // P = exp(z - M) as P_hi | P_lo rows (P_hi in columns 0 .. NH-1, P_lo in NH .. 2NH-1 of
      // the entry's 128-byte row), the FP8 row scale on the weights; per-head sums of P
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) {
        float pe[8];
        uint32_t hi[4], lw[4];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float M = sh.mref[hb + 8 * gi + k];
          pe[k] = on ? __expf(z[8 * gi + k] - (M == -INFINITY ? 0.f : M)) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float a0 = pe[2 * k] * rs, a1 = pe[2 * k + 1] * rs;
          hi[k] = pack_bf16x2(a0, a1);
          lw[k] = pack_bf16x2(a0 - bf16_lo(hi[k]), a1 - bf16_hi(hi[k]));
        }
        const int ci = hb / 8 + gi;
        if (ok) {  // (after a failed wait P may still be read by an earlier second GEMM)
          *reinterpret_cast<uint4*>(ps + e * 128 + ((ci ^ (e & 7)) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(ps + e * 128 + (((NH / 8 + ci) ^ (e & 7)) << 4)) =
              make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        group_reduce8<false>(pe);
        if ((lane & 3) == 0) sh.red_sum[qw][hb + 8 * gi + lh] = pe[0];
      }
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      tc05::fence_before();
      named_bar(1, 256);
      if (qw == 0 && lane < HALF) {
        const int h = hb + lane;
        sh.lsum[h] = sh.lsum[h] * sh.alpha[h] +
                     ((sh.red_sum[0][h] + sh.red_sum[1][h]) + (sh.red_sum[2][h] + sh.red_sum[3][h]));
      }
      if (ok && sw == 0 && lane == 0) tc05::mbar_arrive(&sh.p_full);
    }
    if (!ok && !sh.timeout) report_timeout_attn(&sh.timeout, p.dev_status);
    // ------------------------------------------------------------ output
    const bool live = __all_sync(0xffffffffu, ok && pipe_wait(&sh.o_done, 0, &sh.timeout));
    if (ok && !live && lane == 0 && !sh.timeout) report_timeout_attn(&sh.timeout, p.dev_status);
    tc05::fence_after();
    named_bar(1, 256);  // the last tile's running sums are final
    if (sw == 0) {
      // the sink joins the denominator: o = O e^{M - Mf} / (l e^{M - Mf} + e^{sink - Mf})
      const int h = lane;
      const float M = sh.mref[h], sk = __ldg(p.sink + h0 + h);
      const float Mf = fmaxf(M, sk);
      const float so = M == -INFINITY ? 0.f : __expf(M - Mf);
      const float es = __expf(sk - Mf);
      const float den = sh.lsum[h] * so + es;
      sh.alpha[h] = so / den;
      if (p.sink_mass) p.sink_mass[(size_t)row * kHeads + h0 + h] = es / den;
    }
    named_bar(1, 256);
    if (live) {
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * (sw >> 2) + cc;
        const int d = 128 * c + 32 * qw + lane;
        uint32_t v[32], v2[32];
        const uint32_t ta = lane_base + NO * c;
        tc05::tmem_ld32(ta, v);
        tc05::tmem_ld32(ta + 32, v2);
        tc05::tmem_ld_wait();
        float o[NH];
#pragma unroll
        for (int k = 0; k < NH; ++k) o[k] = (__uint_as_float(v[k]) + __uint_as_float(v2[k])) * sh.alpha[k];
        if (d >= kHeadDim - kRopeDim) {
          // turned back by -position: pairs (448 + 2i, 449 + 2i) sit in adjacent lanes
          const int i = (d - (kHeadDim - kRopeDim)) >> 1;
          const float cn = sh.cs[i], sn = sh.cs[32 + i];
          const bool even = (d & 1) == 0;
#pragma unroll
          for (int k = 0; k < NH; ++k) {
            const float other = __shfl_xor_sync(0xffffffffu, o[k], 1);
            o[k] = even ? o[k] * cn + other * sn : o[k] * cn - other * sn;
          }
        }
        const size_t at = ((size_t)row * kHeads + h0) * kHeadDim + d;
#pragma unroll
        for (int k = 0; k < NH; ++k) {
          if (p.out_bf16) static_cast<__nv_bfloat16*>(p.out)[at + (size_t)k * kHeadDim] = __float2bfloat16_rn(o[k]);
          else static_cast<float*>(p.out)[at + (size_t)k * kHeadDim] = o[k];
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc05::fence_before();
  __syncthreads();  // the MMA thread saw every MMA complete
  if (warp == 0) {
    tc05::fence_after();
    tc05::tmem_dealloc(tmem, kCols);
  }
}

// Merges the tiles of a row for one head: the log-sum-exp over the tiles plus the sink (in the
// denominator only), the normalised sum of the tiles' outputs, and the inverse RoPE on dims
// 448..511.  One warp per (row, head) item, lane l holding dims 4l + 128j (j = 0..3); a grid
// of one block per SM (16 warps) walks the items, one round for up to 16 items per SM (the
// merge is bound by the latency of its L2 reads, so the items should all be in flight at
// once).  A warp issues the loads of all of an item's tile partials (up to kCombPre tiles at
// once) and its tile statistics together, then forms the factors; the rotary cos / sin of its
// row come from one lane per pair by shuffles.
constexpr int kCombWarps = 16;
constexpr int kCombPre = 6;    // tiles whose partials a lane holds at once
__global__ void __launch_bounds__(kCombWarps * 32) attn_combine_kernel(const AttnParams p, int n_tiles) {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");  // the tiles' partials are complete
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int n_items = p.n_rows * kHeads;
  // items interleaved over the blocks (item = block + gridDim.x * k): few items spread over many
  // SMs, whose load bandwidth the partials' loads need
#pragma unroll 1
  for (int item = blockIdx.x + gridDim.x * (threadIdx.x >> 5); item < n_items; item += gridDim.x * kCombWarps) {
    const int row = item / kHeads, h = item % kHeads;
    // tile t of the row: part t / T, tile t % T of that part (one part: T = n_tiles)
    const int T = p.part_tiles > 0 ? p.part_tiles : n_tiles;
    auto tile_o = [&](int t) -> const float* {
      return p.part_o + (size_t)(t / T) * p.part_stride_o + (((size_t)row * T + t % T) * kHeads + h) * kHeadDim +
             4 * lane;
    };
    float4 v[kCombPre][4];
#pragma unroll
    for (int t = 0; t < kCombPre; ++t)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        v[t][j] = t < n_tiles ? __ldcg(reinterpret_cast<const float4*>(tile_o(t) + 128 * j))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
    // this lane's tile statistics (lane t: tile t) and the row's rotary pair `lane`
    float m = -INFINITY, l = 0.f;
    if (lane < n_tiles) {
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml + (size_t)(lane / T) * p.part_stride_ml) +
                               ((size_t)row * T + lane % T) * kHeads + h);
      m = ml.x;
      l = ml.y;
    }
    float cs_c, cs_s;  // turned back by -position: cos, -sin of the row's angles
    if (p.rope_cs != nullptr) {
      cs_c = __ldcg(p.rope_cs + (size_t)row * kRopeDim + lane);
      cs_s = -__ldcg(p.rope_cs + (size_t)row * kRopeDim + 32 + lane);
    } else {
      rope_cs(p.q_pos[row], p.inv_freq[lane], -1.f, &cs_c, &cs_s);
    }
    const float sk = __ldg(p.sink + h);
    const float M = fmaxf(warp_max(m), sk);
    const float f = m == -INFINITY ? 0.f : __expf(m - M);
    const float den = warp_sum(l * f) + __expf(sk - M);
    const float inv_den = 1.f / den;
    if (lane == 0 && p.sink_mass) p.sink_mass[(size_t)row * kHeads + h] = __expf(sk - M) * inv_den;
    float4 acc[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int t = 0; t < kCombPre; ++t) {
      const float ft = __shfl_sync(0xffffffffu, f, t);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[j].x = fmaf(ft, v[t][j].x, acc[j].x);
        acc[j].y = fmaf(ft, v[t][j].y, acc[j].y);
        acc[j].z = fmaf(ft, v[t][j].z, acc[j].z);
        acc[j].w = fmaf(ft, v[t][j].w, acc[j].w);
      }
    }
#pragma unroll 1
    for (int t = kCombPre; t < n_tiles; ++t) {  // rows with more tiles than a lane holds
      const float ft = __shfl_sync(0xffffffffu, f, t);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 x = __ldcg(reinterpret_cast<const float4*>(tile_o(t) + 128 * j));
        acc[j].x = fmaf(ft, x.x, acc[j].x);
        acc[j].y = fmaf(ft, x.y, acc[j].y);
        acc[j].z = fmaf(ft, x.z, acc[j].z);
        acc[j].w = fmaf(ft, x.w, acc[j].w);
      }
    }
    // inverse rotation: dims 448 + 4(l - 16) .. of chunk j = 3 hold pairs 2(l - 16) and 2(l - 16) + 1
    const int pa = 2 * (lane & 15), pb = pa + 1;
    const float ca = __shfl_sync(0xffffffffu, cs_c, pa), sa = __shfl_sync(0xffffffffu, cs_s, pa);
    const float cb = __shfl_sync(0xffffffffu, cs_c, pb), sb = __shfl_sync(0xffffffffu, cs_s, pb);
    float4 o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = make_float4(acc[j].x * inv_den, acc[j].y * inv_den, acc[j].z * inv_den, acc[j].w * inv_den);
    if (lane >= 16) {
      const float x0 = o[3].x, y0 = o[3].y, x1 = o[3].z, y1 = o[3].w;
      o[3] = make_float4(x0 * ca - y0 * sa, x0 * sa + y0 * ca, x1 * cb - y1 * sb, x1 * sb + y1 * cb);
    }
    const size_t at = ((size_t)row * kHeads + h) * kHeadDim + 4 * lane;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (p.out_bf16) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(o[j].x, o[j].y), hi = __floats2bfloat162_rn(o[j].z, o[j].w);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + at + 128 * j) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
      } else {
        *reinterpret_cast<float4*>(static_cast<float*>(p.out) + at + 128 * j) = o[j];
      }
    }
  }
}

// The row kernel runs its tiles one after another in one block, a chain per tile that the
// tile kernel runs in parallel blocks: measured slower for every decode workload (B=32
// 0.134-0.138 against 0.118 ms; tiny 54-57 against 34 us) and no faster for the prefill
// chunk, whose partials it saves (2.53 ms either way), so it is chosen only through
// CSA2_TUNE_ATTN_ROWS.
bool use_row_kernel(const AttnParams& p, int n_split) {
  (void)p;
  (void)n_split;
  return false;
}
int row_kernel_heads(const AttnParams& p) {
  (void)p;
  return 32;
}

}  // namespace

int attn_smem_bytes() { return kAttnSmemBytes; }

cudaError_t launch_sparse_attn(const AttnParams& p, int n_split, cudaStream_t stream) {
  if (p.n_rows == 0) return cudaSuccess;
  const int rows_mode = tuning(CSA2_TUNE_ATTN_ROWS);
  // Many rows (a prefill chunk), bf16 latents and window: the pipelined row kernel, two
  // blocks per row (32 heads each).  With fewer rows than two per SM its serial tiles cost
  // more latency than the tile kernel's parallel ones.
  const bool pipe_ok = p.lat_fmt == CSA2_BF16 && (p.swa_fmt == CSA2_BF16 || p.window == 0) && p.range_count == 0;
  if (pipe_ok && (rows_mode == 4 || (rows_mode == 0 && p.n_rows >= 2 * device_sm_count()))) {
    cudaError_t e = cudaFuncSetAttribute(attn_pipe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         pipe_smem_bytes());
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_rows, kHeads / kPipeNH);
    cfg.blockDim = dim3(kPipeThreads);
    cfg.dynamicSmemBytes = pipe_smem_bytes();
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_pipe_kernel, p);
  }
  if (rows_mode == 2 || rows_mode == 3 || (rows_mode == 0 && use_row_kernel(p, n_split))) {
    // whole rows per block, no partials and no merge
    const int nh = rows_mode == 3 ? 16 : rows_mode == 2 ? 32 : row_kernel_heads(p);
    auto kern = nh == 16 ? attn_row_kernel<16> : attn_row_kernel<32>;
    const int smem = nh == 16 ? row_smem_bytes<16>() : row_smem_bytes<32>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_rows, kHeads / nh);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
  }
  const cudaError_t e = launch_attn_tiles(p, n_split, stream);
  if (e != cudaSuccess) return e;
  return launch_attn_merge(p, n_split, stream);
}

// Both kernels may start before their predecessor in the stream has finished (programmatic
// dependent launch); each waits for it where it reads its results.
cudaError_t launch_attn_tiles(const AttnParams& p, int n_split, cudaStream_t stream) {
  if (p.n_rows == 0) return cudaSuccess;
  // Heads per block: all 64, or 32 / 16 where rows x tiles blocks would leave most SMs idle
  // (the tile chain then runs on half / a quarter of the heads, in parallel).
  const int sms = device_sm_count();
  const long long tiles = (long long)p.n_rows * n_split;
  const int nh = tiles * 4 <= sms ? 16 : tiles * 2 <= sms ? 32 : 64;
  auto kern = nh == 16 ? attn_tc05_kernel<16> : nh == 32 ? attn_tc05_kernel<32> : attn_tc05_kernel<64>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_rows, n_split * (kHeads / nh));
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = kAttnSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_attn_merge(const AttnParams& p, int n_tiles, cudaStream_t stream) {
  if (p.n_rows == 0) return cudaSuccess;
  if (n_tiles < 1 || n_tiles > 32) return cudaErrorInvalidValue;  // one lane per tile's statistics
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  const int items = p.n_rows * kHeads;
  cfg.gridDim = dim3(std::min(device_sm_count(), items));
  cfg.blockDim = dim3(kCombWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_combine_kernel, p, n_tiles);
}

}  // namespace csa2
