// Sparse shared-latent MQA of one query row over its selected latents plus its sliding
// window, with one sink logit per head ("DeepSeek V4 Inside", CSA core attention and
// eq. (27); "Every layer, connected", "The query and output paths").
//
// Split-K flash decode: the K + W attended entries of a row are cut into tiles of 64; a
// thread block (16 warps) handles a contiguous range of tiles of one row and keeps, per
// head, the running max m, the running sum l and the unnormalised output O (64 x 512 fp32,
// 64 registers per thread).  Each tile is gathered into shared memory (bf16 rows by
// cp.async; FP4 latents and FP8 window rows are widened to bf16 in registers on the way,
// which is exact), then
//   S = q' K^T   on the tensor cores in bf16 (64 heads x 64 rows x 512), fp32 accumulate;
//   P = exp(S - m) written as fp16 (10-bit mantissa keeps the rounding of P at ~2^-12);
//   O = alpha O + P V  in fp16 x fp16 -> fp32 (V widened from the bf16 tile in registers).
// The FP8 window rows' scale multiplies their logits and their weights in P.  A second
// kernel merges the splits (log-sum-exp), adds the sink to the denominator, normalises and
// turns the output's rotary coordinates back by -position.  With one split per row the
// first kernel finishes the row itself.
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace csa2 {

namespace {

constexpr int kAttnThreads = 256;  // 8 warps
constexpr int kTile = 64;          // attended entries per tile
constexpr int kHG = 16;            // heads per block (one m16 MMA tile)
constexpr int kQBytes = kHG * kHeadDim * 2;     // 16 KB
constexpr int kKVBytes = kTile * kHeadDim * 2;  // 64 KB per stage
constexpr int kPBytes = kHG * kTile * 2;        // 2 KB
constexpr int kStages = 3;                      // gather pipeline depth (tiles in flight)
constexpr int kMetaSlots = kStages + 1;         // tile sources, prepared one iteration ahead

struct TileMeta {
  const uint8_t* ptr[kTile];   // first byte of each entry's row (codes for FP formats)
  const uint8_t* sptr[kTile];  // FP4 group scales
  float rs[kTile];             // FP8 row scale (1 otherwise)
  int fmt[kTile];              // storage format, -1 = masked entry
};

struct AttnSmem {
  TileMeta meta[kMetaSlots];
  float red_max[4][kHG];
  float red_sum[4][kHG];
  float cs[kRopeDim];  // cos (0..31) and sin (32..63) of the row's rotary angles
};
constexpr int kAttnSmemBytes = kQBytes + kStages * kKVBytes + kPBytes + (int)sizeof(AttnSmem);

// Byte offset of 16-byte chunk `c` of row `r` in a tile with 1024-byte rows: the low three
// chunk bits are XOR-ed with the row so that 8 rows at the same chunk hit 8 bank groups.
__device__ __forceinline__ int swz1k(int r, int c) { return r * 1024 + ((c ^ (r & 7)) << 4); }
// Same for the P tile (128-byte rows of 64 fp16).
__device__ __forceinline__ int swzp(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ float e2m1_level(uint32_t nib) {
  // magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6; bit 3 is the sign
  const uint32_t e = (nib >> 1) & 3u, m = nib & 1u;
  const float mag = e == 0 ? 0.5f * (float)m : (1.0f + 0.5f * (float)m) * (float)(1u << (e - 1));
  return (nib & 8u) ? -mag : mag;
}
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  const uint32_t e = (code >> 3) & 15u, m = code & 7u;
  const float mag = e == 0 ? (float)m * 0.001953125f /* 2^-9 */ : ldexpf(1.0f + 0.125f * (float)m, (int)e - 7);
  return (code & 0x80u) ? -mag : mag;
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

__device__ __forceinline__ EntrySrc entry_source(const AttnParams& p, int row, int b, long long qp, long long lo,
                                                 long long pos0, int e) {
  EntrySrc s{nullptr, nullptr, 1.f, CSA2_BF16, false};
  if (e < p.K) {
    const int rec = __ldg(p.idx + (size_t)row * p.K + e);
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
  } else if (e < p.K + p.window) {
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

// Source of every entry of tile `tile` (threads 0..63, one entry each).
__device__ __forceinline__ void tile_meta(const AttnParams& p, TileMeta& m, int row, int b, long long qp, long long lo,
                                          long long pos0, int tile) {
  if (threadIdx.x < kTile) {
    const int r = threadIdx.x;
    const EntrySrc s = entry_source(p, row, b, qp, lo, pos0, tile * kTile + r);
    m.ptr[r] = s.valid ? s.ptr : nullptr;
    m.sptr[r] = s.sptr;
    m.rs[r] = s.rs;
    m.fmt[r] = s.valid ? s.fmt : -1;
  }
}

// Gathers one tile into a KV stage (64 rows x 512 bf16, swizzled).  bf16 rows go by cp.async,
// a warp copying 512 contiguous bytes per instruction; FP4 latents and FP8 window rows are
// widened to bf16 in registers (exact) by four threads per row.
__device__ __forceinline__ void load_tile(const TileMeta& m, uint8_t* kv, const void* any_valid) {
  const int t = threadIdx.x;
#pragma unroll 4
  for (int k = 0; k < kTile / 4; ++k) {
    const int r = 4 * k + (t >> 6), c = t & 63;
    const int f = m.fmt[r];
    if (f == CSA2_BF16 || f < 0) {
      const uint8_t* src = f < 0 ? reinterpret_cast<const uint8_t*>(any_valid) : m.ptr[r];
      cp_async16(kv + swz1k(r, c), src + c * 16, f >= 0);
    }
  }
  const int r = t >> 2, quarter = t & 3;  // 128 dims per thread
  const int f = m.fmt[r];
  if (f == CSA2_FP8_E4M3_ROWSCALE) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int d0 = quarter * 128 + half * 64;
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
        *reinterpret_cast<uint4*>(kv + swz1k(r, d0 / 8 + k)) =
            make_uint4(outw[4 * k], outw[4 * k + 1], outw[4 * k + 2], outw[4 * k + 3]);
    }
  } else if (f == CSA2_FP4_E2M1_G32 || f == CSA2_FP4_E2M1_G16) {
    const int gsz = f == CSA2_FP4_E2M1_G32 ? 32 : 16;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int d0 = quarter * 128 + half * 64;
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
            const int ch = d0 + h2 * 32 + k * 8 + byte * 2;  // even channel of this byte
            const float sc = e4m3_value(__ldg(m.sptr[r] + ch / gsz));
            const uint32_t code = (w4[k] >> (8 * byte)) & 0xffu;
            outw[h2 * 16 + k * 4 + byte] = pack_bf16x2(e2m1_level(code & 15u) * sc, e2m1_level(code >> 4) * sc);
          }
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k)
        *reinterpret_cast<uint4*>(kv + swz1k(r, d0 / 8 + k)) =
            make_uint4(outw[4 * k], outw[4 * k + 1], outw[4 * k + 2], outw[4 * k + 3]);
    }
  }
}

// One block: query row blockIdx.z, heads 16*blockIdx.y .. +15, split blockIdx.x of the row's
// tiles.  Gathers run kStages tiles ahead.  Warps 0..3: QK for rows 16w..16w+15 of each tile
// and the softmax; all 8 warps: PV for dims 64w..64w+63.
__global__ void __launch_bounds__(kAttnThreads, 1) attn_hg_kernel(const AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* Qs = smem;
  uint8_t* KV = smem + kQBytes;
  uint8_t* Ps = KV + kStages * kKVBytes;
  AttnSmem& sm = *reinterpret_cast<AttnSmem*>(Ps + kPBytes);

  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int row = blockIdx.z, hg = blockIdx.y, split = blockIdx.x, n_split = gridDim.x;
  const int b = p.seq_of_row[row];
  const long long qp = p.q_pos[row];
  const long long pos0 = p.swa_pos0[b];
  const long long lo = max(qp - (long long)p.window + 1, pos0);
  const int n_tiles = (p.K + p.window + kTile - 1) / kTile;
  const int t0 = (int)(((long long)n_tiles * split) / n_split);
  const int t1 = (int)(((long long)n_tiles * (split + 1)) / n_split);

  rope_table(sm.cs, p, qp, 1.f);
#pragma unroll
  for (int k = 0; k < kStages; ++k)
    if (t0 + k < t1) tile_meta(p, sm.meta[(t0 + k) % kMetaSlots], row, b, qp, lo, pos0, t0 + k);
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kStages - 1; ++k) {
    if (t0 + k < t1) load_tile(sm.meta[(t0 + k) % kMetaSlots], KV + ((t0 + k) % kStages) * kKVBytes, p.q);
    cp_async_commit();
  }
  // ---- q' = RoPE(q) for this block's 16 heads (coalesced: consecutive threads, consecutive chunks)
  {
    const uint4* qsrc = reinterpret_cast<const uint4*>(p.q) + ((size_t)row * kHeads + kHG * hg) * (kHeadDim / 8);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int idx = k * kAttnThreads + tid, h = idx >> 6, ch = idx & 63;
      uint4 v = __ldg(qsrc + idx);
      if (ch >= 56) {
        uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = (ch - 56) * 4 + j;  // rotary pair index
          const float x = bf16_lo(w4[j]), y = bf16_hi(w4[j]);
          const float cs = sm.cs[i], sn = sm.cs[32 + i];
          w4[j] = pack_bf16x2(x * cs - y * sn, x * sn + y * cs);
        }
        v = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
      *reinterpret_cast<uint4*>(Qs + swz1k(h, ch)) = v;
    }
  }

  float m_run[2] = {-INFINITY, -INFINITY};  // heads g, g+8 of the group
  float l_run[2] = {0.f, 0.f};
  float acc_o[8][4];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) acc_o[nt][0] = acc_o[nt][1] = acc_o[nt][2] = acc_o[nt][3] = 0.f;

  const uint32_t qs_u = smem_u32(Qs), ps_u = smem_u32(Ps);
  const int mi = lane >> 3, ri = lane & 7;
  for (int t = t0; t < t1; ++t) {
    const int st = t % kStages;
    uint8_t* kv = KV + st * kKVBytes;
    {
      const int tn = t + kStages - 1;  // sources of tn were prepared one iteration ago
      if (tn < t1) load_tile(sm.meta[tn % kMetaSlots], KV + (tn % kStages) * kKVBytes, p.q);
      cp_async_commit();
    }
    cp_async_wait<kStages - 1>();
    __syncthreads();
    const uint32_t kv_u = smem_u32(kv);
    const TileMeta& md = sm.meta[t % kMetaSlots];

    float alpha[2] = {1.f, 1.f};
    if (wid < 4) {
      // ---- S = q' K^T: 16 heads x rows 16*wid .. +15 (two 8-row MMA tiles, two chains each)
      float sa[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a) sa[a][0] = sa[a][1] = sa[a][2] = sa[a][3] = 0.f;
      const int qh = ri + (mi & 1) * 8;
      const int kr = 16 * wid + ri + (mi >> 1) * 8;
#pragma unroll
      for (int ks = 0; ks < kHeadDim / 16; ++ks) {
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        ldsm_x4(a0, a1, a2, a3, qs_u + swz1k(qh, 2 * ks + (mi >> 1)));
        ldsm_x4(b0, b1, b2, b3, kv_u + swz1k(kr, 2 * ks + (mi & 1)));
        mma_bf16(sa[(ks & 1) * 2 + 0], a0, a1, a2, a3, b0, b1);
        mma_bf16(sa[(ks & 1) * 2 + 1], a0, a1, a2, a3, b2, b3);
      }
      // sacc[nt][e]: n-tile nt = rows 16*wid + 8*nt .. ; e as in the MMA C fragment
      float sacc[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[nt][e] = sa[nt][e] + sa[2 + nt][e];
      float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = 16 * wid + 8 * nt + 2 * c + (e & 1);
          const float z = md.fmt[r] >= 0 ? sacc[nt][e] * p.scale * md.rs[r] : -INFINITY;
          sacc[nt][e] = z;
          tmax[e >> 1] = fmaxf(tmax[e >> 1], z);
        }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        tmax[hh] = fmaxf(tmax[hh], __shfl_xor_sync(0xffffffffu, tmax[hh], 1));
        tmax[hh] = fmaxf(tmax[hh], __shfl_xor_sync(0xffffffffu, tmax[hh], 2));
      }
      if (c == 0) {
        sm.red_max[wid][g] = tmax[0];
        sm.red_max[wid][g + 8] = tmax[1];
      }
      asm volatile("bar.sync 2, 128;\n" ::: "memory");
      float m_use[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int h = g + 8 * hh;
        const float tm = fmaxf(fmaxf(sm.red_max[0][h], sm.red_max[1][h]), fmaxf(sm.red_max[2][h], sm.red_max[3][h]));
        const float m_new = fmaxf(m_run[hh], tm);
        m_use[hh] = m_new == -INFINITY ? 0.f : m_new;
        alpha[hh] = m_run[hh] == -INFINITY ? 0.f : __expf(m_run[hh] - m_use[hh]);
        m_run[hh] = m_new;
      }
      float psum[2] = {0.f, 0.f};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        float pe[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          pe[e] = __expf(sacc[nt][e] - m_use[e >> 1]);
          psum[e >> 1] += pe[e];
        }
        const int r = 16 * wid + 8 * nt + 2 * c;
        const float rs0 = md.rs[r], rs1 = md.rs[r + 1];
        // P[h][r], P[h][r+1] as fp16 pairs; the FP8 row scale multiplies the weights
        *reinterpret_cast<uint32_t*>(Ps + swzp(g, r >> 3) + (r & 7) * 2) = pack_f16x2(pe[0] * rs0, pe[1] * rs1);
        *reinterpret_cast<uint32_t*>(Ps + swzp(g + 8, r >> 3) + (r & 7) * 2) = pack_f16x2(pe[2] * rs0, pe[3] * rs1);
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        psum[hh] += __shfl_xor_sync(0xffffffffu, psum[hh], 1);
        psum[hh] += __shfl_xor_sync(0xffffffffu, psum[hh], 2);
      }
      if (c == 0) {
        sm.red_sum[wid][g] = psum[0];
        sm.red_sum[wid][g + 8] = psum[1];
      }
    }
    __syncthreads();
    // every warp: the running statistics of heads g, g+8 (identical in all warps)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int h = g + 8 * hh;
      if (wid >= 4) {
        const float tm = fmaxf(fmaxf(sm.red_max[0][h], sm.red_max[1][h]), fmaxf(sm.red_max[2][h], sm.red_max[3][h]));
        const float m_new = fmaxf(m_run[hh], tm);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        alpha[hh] = m_run[hh] == -INFINITY ? 0.f : __expf(m_run[hh] - m_use);
        m_run[hh] = m_new;
      }
      const float ts = (sm.red_sum[0][h] + sm.red_sum[1][h]) + (sm.red_sum[2][h] + sm.red_sum[3][h]);
      l_run[hh] = l_run[hh] * alpha[hh] + ts;
    }
    // ---- O = alpha O + P V for dims 64*wid .. +63
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      acc_o[nt][0] *= alpha[0];
      acc_o[nt][1] *= alpha[0];
      acc_o[nt][2] *= alpha[1];
      acc_o[nt][3] *= alpha[1];
    }
#pragma unroll
    for (int ks = 0; ks < kTile / 16; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(a0, a1, a2, a3, ps_u + swzp(ri + (mi & 1) * 8, 2 * ks + (mi >> 1)));
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t vb[4];
        const int vr = 16 * ks + ri + (mi & 1) * 8;
        const int vc = (64 * wid + 16 * np) / 8 + (mi >> 1);
        ldsm_x4_t(vb[0], vb[1], vb[2], vb[3], kv_u + swz1k(vr, vc));
#pragma unroll
        for (int k = 0; k < 4; ++k) vb[k] = bf16x2_to_f16x2(vb[k]);
        mma_f16(acc_o[2 * np], a0, a1, a2, a3, vb[0], vb[1]);
        mma_f16(acc_o[2 * np + 1], a0, a1, a2, a3, vb[2], vb[3]);
      }
    }
    if (t + kStages < t1) tile_meta(p, sm.meta[(t + kStages) % kMetaSlots], row, b, qp, lo, pos0, t + kStages);
    __syncthreads();
  }
  cp_async_wait<0>();

  const int h_lo = kHG * hg + g, h_hi = h_lo + 8;  // absolute heads of this thread
  if (n_split == 1) {
    // ---- finish the row: sink in the denominator, normalise, inverse RoPE
    float f[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const float sk = __ldg(p.sink + (hh ? h_hi : h_lo));
      const float M = fmaxf(m_run[hh], sk);
      const float em = m_run[hh] == -INFINITY ? 0.f : __expf(m_run[hh] - M);
      const float den = l_run[hh] * em + __expf(sk - M);
      f[hh] = em / den;
      if (p.sink_mass && wid == 0 && c == 0) p.sink_mass[(size_t)row * kHeads + (hh ? h_hi : h_lo)] = __expf(sk - M) / den;
    }
    rope_table(sm.cs, p, qp, -1.f);
    __syncthreads();
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float* orow = p.out + ((size_t)row * kHeads + (hh ? h_hi : h_lo)) * kHeadDim;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int d = 64 * wid + 8 * nt + 2 * c;
        float x = acc_o[nt][2 * hh] * f[hh], y = acc_o[nt][2 * hh + 1] * f[hh];
        if (d >= kHeadDim - kRopeDim) {
          const int i = (d - (kHeadDim - kRopeDim)) >> 1;
          const float cs = sm.cs[i], sn = sm.cs[32 + i];
          const float xr = x * cs - y * sn, yr = x * sn + y * cs;
          x = xr;
          y = yr;
        }
        *reinterpret_cast<float2*>(orow + d) = make_float2(x, y);
      }
    }
    return;
  }
  // ---- partial results of this split
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    float* po = p.part_o + (((size_t)row * n_split + split) * kHeads + (hh ? h_hi : h_lo)) * kHeadDim;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int d = 64 * wid + 8 * nt + 2 * c;
      *reinterpret_cast<float2*>(po + d) = make_float2(acc_o[nt][2 * hh], acc_o[nt][2 * hh + 1]);
    }
  }
  if (wid == 0 && c == 0) {
    float* pm = p.part_ml + ((size_t)row * n_split + split) * kHeads * 2;
    pm[2 * h_lo] = m_run[0];
    pm[2 * h_lo + 1] = l_run[0];
    pm[2 * h_hi] = m_run[1];
    pm[2 * h_hi + 1] = l_run[1];
  }
}

// Merges the splits of one row for 4 heads: log-sum-exp over splits plus the sink,
// normalisation, inverse RoPE on dims 448..511.  Thread -> (head h0 + tid/32, 16 dims).
__global__ void __launch_bounds__(128) attn_combine_kernel(const AttnParams p, int n_split) {
  __shared__ float fac[4][64];  // per head: weight of each split (n_split <= 64)
  __shared__ float inv_den[4];
  const int row = blockIdx.x, hl = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * 4 + hl;
  const long long qp = p.q_pos[row];
  {
    // warp hl: per-split statistics of head h, two splits per lane
    const float sk = __ldg(p.sink + h);
    float m[2], l[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int s = lane + 32 * k;
      m[k] = -INFINITY;
      l[k] = 0.f;
      if (s < n_split) {
        const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + (((size_t)row * n_split + s) * kHeads + h) * 2);
        m[k] = ml.x;
        l[k] = ml.y;
      }
    }
    const float M = fmaxf(warp_max(fmaxf(m[0], m[1])), sk);
    float f[2], den = 0.f;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      f[k] = m[k] == -INFINITY ? 0.f : __expf(m[k] - M);
      den += l[k] * f[k];
      const int s = lane + 32 * k;
      if (s < n_split) fac[hl][s] = f[k];
    }
    den = warp_sum(den) + __expf(sk - M);
    if (lane == 0) {
      inv_den[hl] = 1.f / den;
      if (p.sink_mass) p.sink_mass[(size_t)row * kHeads + h] = __expf(sk - M) / den;
    }
  }
  __syncthreads();
  const int d0 = lane * 16;
  float4 acc[4] = {};
  const float* base = p.part_o + ((size_t)row * n_split * kHeads + h) * kHeadDim + d0;
  const size_t split_stride = (size_t)kHeads * kHeadDim;
  for (int s = 0; s < n_split; ++s) {
    const float4* src = reinterpret_cast<const float4*>(base + s * split_stride);
    const float f = fac[hl][s];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 v = __ldg(src + k);
      acc[k].x = fmaf(f, v.x, acc[k].x);
      acc[k].y = fmaf(f, v.y, acc[k].y);
      acc[k].z = fmaf(f, v.z, acc[k].z);
      acc[k].w = fmaf(f, v.w, acc[k].w);
    }
  }
  const float inv = inv_den[hl];
  float* dst = p.out + ((size_t)row * kHeads + h) * kHeadDim + d0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float v[4] = {acc[k].x * inv, acc[k].y * inv, acc[k].z * inv, acc[k].w * inv};
    const int d = d0 + 4 * k;
    if (d >= kHeadDim - kRopeDim) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int pi = (d + 2 * j - (kHeadDim - kRopeDim)) >> 1;
        float c, sn;
        rope_cs(qp, p.inv_freq[pi], -1.f, &c, &sn);
        const float x = v[2 * j], y = v[2 * j + 1];
        v[2 * j] = x * c - y * sn;
        v[2 * j + 1] = x * sn + y * c;
      }
    }
    *reinterpret_cast<float4*>(dst + 4 * k) = make_float4(v[0], v[1], v[2], v[3]);
  }
}

}  // namespace

int attn_smem_bytes() { return kAttnSmemBytes; }

cudaError_t launch_sparse_attn(const AttnParams& p, int n_split, cudaStream_t stream) {
  if (p.n_rows == 0) return cudaSuccess;
  cudaError_t e =
      cudaFuncSetAttribute(attn_hg_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmemBytes);
  if (e != cudaSuccess) return e;
  attn_hg_kernel<<<dim3(n_split, kHeads / kHG, p.n_rows), kAttnThreads, kAttnSmemBytes, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess || n_split == 1) return e;
  attn_combine_kernel<<<dim3(p.n_rows, kHeads / 4), 128, 0, stream>>>(p, n_split);
  return cudaGetLastError();
}

}  // namespace csa2
