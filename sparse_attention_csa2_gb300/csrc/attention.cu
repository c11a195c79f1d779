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

constexpr int kAttnThreads = 512;
constexpr int kTile = 64;
constexpr int kQBytes = kHeads * kHeadDim * 2;      // 64 KB
constexpr int kKVBytes = kTile * kHeadDim * 2;      // 64 KB per stage
constexpr int kPBytes = kHeads * kTile * 2;         // 8 KB

struct AttnSmem {
  float red_max[4][kHeads];
  float red_sum[4][kHeads];
  float alpha[kHeads];
  float rowscale[2][kTile];
  int rowvalid[2][kTile];
  float cs[kRopeDim];  // cos (0..31) and sin (32..63) of the row's rotary angles
};
constexpr int kAttnSmemBytes = kQBytes + 2 * kKVBytes + kPBytes + (int)sizeof(AttnSmem);

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

// Gathers tile `tile` of the row into KV stage `kv` (64 rows x 512 bf16, swizzled).
// Thread -> (row = tid/8, part = tid%8); part covers dims 64*part .. 64*part+63.
__device__ __forceinline__ void load_tile(const AttnParams& p, AttnSmem& sm, uint8_t* kv, int stage, int row,
                                          int b, long long qp, long long lo, long long pos0, int tile) {
  const int r = threadIdx.x >> 3, part = threadIdx.x & 7;
  const EntrySrc s = entry_source(p, row, b, qp, lo, pos0, tile * kTile + r);
  if (part == 0) {
    sm.rowvalid[stage][r] = s.valid;
    sm.rowscale[stage][r] = s.rs;
  }
  if (!s.valid || s.fmt == CSA2_BF16) {
    const uint8_t* src = s.valid ? s.ptr : reinterpret_cast<const uint8_t*>(p.q);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = part + 8 * k;
      cp_async16(kv + swz1k(r, c), src + c * 16, s.valid);
    }
    return;
  }
  uint32_t outw[32];  // 64 bf16 of dims 64*part ..
  if (s.fmt == CSA2_FP8_E4M3_ROWSCALE) {
    const uint4* src = reinterpret_cast<const uint4*>(s.ptr + part * 64);
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
  } else {
    const int gsz = s.fmt == CSA2_FP4_E2M1_G32 ? 32 : 16;
    const uint4* src = reinterpret_cast<const uint4*>(s.ptr + part * 32);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 v = __ldg(src + h);
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
#pragma unroll
        for (int byte = 0; byte < 4; ++byte) {
          const int ch = part * 64 + h * 32 + k * 8 + byte * 2;  // even channel of this byte
          const float sc = e4m3_value(__ldg(s.sptr + ch / gsz));
          const uint32_t code = (w4[k] >> (8 * byte)) & 0xffu;
          outw[h * 16 + k * 4 + byte] = pack_bf16x2(e2m1_level(code & 15u) * sc, e2m1_level(code >> 4) * sc);
        }
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int c = part * 8 + k;
    *reinterpret_cast<uint4*>(kv + swz1k(r, c)) =
        make_uint4(outw[4 * k], outw[4 * k + 1], outw[4 * k + 2], outw[4 * k + 3]);
  }
}

__global__ void __launch_bounds__(kAttnThreads, 1) attn_split_kernel(const AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* Qs = smem;
  uint8_t* KV = smem + kQBytes;
  uint8_t* Ps = KV + 2 * kKVBytes;
  AttnSmem& sm = *reinterpret_cast<AttnSmem*>(Ps + kPBytes);

  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int row = blockIdx.y, split = blockIdx.x, n_split = gridDim.x;
  const int b = p.seq_of_row[row];
  const long long qp = p.q_pos[row];
  const long long pos0 = p.swa_pos0[b];
  const long long lo = max(qp - (long long)p.window + 1, pos0);
  const int n_tiles = (p.K + p.window + kTile - 1) / kTile;
  const int t0 = (int)(((long long)n_tiles * split) / n_split);
  const int t1 = (int)(((long long)n_tiles * (split + 1)) / n_split);

  rope_table(sm.cs, p, qp, 1.f);
  if (t0 < t1) load_tile(p, sm, KV, 0, row, b, qp, lo, pos0, t0);
  cp_async_commit();
  __syncthreads();

  // ---- q' = RoPE(q): head h = tid/8, dims 64*part .. ; part 7 holds the rotary dims
  {
    const int h = tid >> 3, part = tid & 7;
    const uint4* src = reinterpret_cast<const uint4*>(p.q) + ((size_t)row * kHeads + h) * (kHeadDim / 8) + part * 8;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint4 v = __ldg(src + k);
      if (part == 7) {
        uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = k * 4 + j;  // rotary pair index
          const float x = bf16_lo(w4[j]), y = bf16_hi(w4[j]);
          const float cs = sm.cs[i], sn = sm.cs[32 + i];
          w4[j] = pack_bf16x2(x * cs - y * sn, x * sn + y * cs);
        }
        v = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
      *reinterpret_cast<uint4*>(Qs + swz1k(h, part * 8 + k)) = v;
    }
  }

  const int hq = 16 * (wid & 3);   // QK: head block of this warp
  const int rq = 16 * (wid >> 2);  // QK: row block of this warp
  float m_run[2] = {-INFINITY, -INFINITY};  // heads hq+g, hq+g+8
  float l_run[2] = {0.f, 0.f};
  float acc_o[4][4][4];
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) acc_o[mt][nt][0] = acc_o[mt][nt][1] = acc_o[mt][nt][2] = acc_o[mt][nt][3] = 0.f;

  const uint32_t qs_u = smem_u32(Qs), ps_u = smem_u32(Ps);
  for (int t = t0; t < t1; ++t) {
    const int stage = (t - t0) & 1;
    uint8_t* kv = KV + stage * kKVBytes;
    if (t + 1 < t1) load_tile(p, sm, KV + (stage ^ 1) * kKVBytes, stage ^ 1, row, b, qp, lo, pos0, t + 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const uint32_t kv_u = smem_u32(kv);

    // ---- S = q' K^T for heads hq..hq+15, rows rq..rq+15
    float sacc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
    {
      const int mi = lane >> 3, ri = lane & 7;
      const int qh = hq + ri + (mi & 1) * 8;
      const int kr = rq + ri + (mi >> 1) * 8;
#pragma unroll 8
      for (int ks = 0; ks < kHeadDim / 16; ++ks) {
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        ldsm_x4(a0, a1, a2, a3, qs_u + swz1k(qh, 2 * ks + (mi >> 1)));
        ldsm_x4(b0, b1, b2, b3, kv_u + swz1k(kr, 2 * ks + (mi & 1)));
        mma_bf16(sacc[0], a0, a1, a2, a3, b0, b1);
        mma_bf16(sacc[1], a0, a1, a2, a3, b2, b3);
      }
    }
    // ---- online softmax over the tile
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = rq + 8 * nt + 2 * c + (e & 1);
        const float z = sm.rowvalid[stage][r] ? sacc[nt][e] * p.scale * sm.rowscale[stage][r] : -INFINITY;
        sacc[nt][e] = z;
        tmax[e >> 1] = fmaxf(tmax[e >> 1], z);
      }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      tmax[hh] = fmaxf(tmax[hh], __shfl_xor_sync(0xffffffffu, tmax[hh], 1));
      tmax[hh] = fmaxf(tmax[hh], __shfl_xor_sync(0xffffffffu, tmax[hh], 2));
    }
    if (c == 0) {
      sm.red_max[wid >> 2][hq + g] = tmax[0];
      sm.red_max[wid >> 2][hq + g + 8] = tmax[1];
    }
    __syncthreads();
    float m_new[2], m_use[2], alpha[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int h = hq + g + 8 * hh;
      const float tm = fmaxf(fmaxf(sm.red_max[0][h], sm.red_max[1][h]), fmaxf(sm.red_max[2][h], sm.red_max[3][h]));
      m_new[hh] = fmaxf(m_run[hh], tm);
      m_use[hh] = m_new[hh] == -INFINITY ? 0.f : m_new[hh];
      alpha[hh] = m_run[hh] == -INFINITY ? 0.f : __expf(m_run[hh] - m_use[hh]);
    }
    float psum[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int r = rq + 8 * nt + 2 * c;
      float pe[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        pe[e] = __expf(sacc[nt][e] - m_use[e >> 1]);
        psum[e >> 1] += pe[e];
      }
      const float rs0 = sm.rowscale[stage][r], rs1 = sm.rowscale[stage][r + 1];
      // P[h][r], P[h][r+1] as fp16 pairs; the FP8 row scale multiplies the weights
      *reinterpret_cast<uint32_t*>(Ps + swzp(hq + g, r >> 3) + (r & 7) * 2) = pack_f16x2(pe[0] * rs0, pe[1] * rs1);
      *reinterpret_cast<uint32_t*>(Ps + swzp(hq + g + 8, r >> 3) + (r & 7) * 2) = pack_f16x2(pe[2] * rs0, pe[3] * rs1);
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      psum[hh] += __shfl_xor_sync(0xffffffffu, psum[hh], 1);
      psum[hh] += __shfl_xor_sync(0xffffffffu, psum[hh], 2);
    }
    if (c == 0) {
      sm.red_sum[wid >> 2][hq + g] = psum[0];
      sm.red_sum[wid >> 2][hq + g + 8] = psum[1];
      if ((wid >> 2) == 0) {
        sm.alpha[hq + g] = alpha[0];
        sm.alpha[hq + g + 8] = alpha[1];
      }
    }
    __syncthreads();
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int h = hq + g + 8 * hh;
      const float ts = sm.red_sum[0][h] + sm.red_sum[1][h] + sm.red_sum[2][h] + sm.red_sum[3][h];
      l_run[hh] = l_run[hh] * alpha[hh] + ts;
      m_run[hh] = m_new[hh];
    }
    // ---- O = alpha O + P V for dims 32*wid .. 32*wid+31, all heads
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const float a_lo = sm.alpha[16 * mt + g], a_hi = sm.alpha[16 * mt + g + 8];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        acc_o[mt][nt][0] *= a_lo;
        acc_o[mt][nt][1] *= a_lo;
        acc_o[mt][nt][2] *= a_hi;
        acc_o[mt][nt][3] *= a_hi;
      }
    }
    {
      const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
      for (int ks = 0; ks < kTile / 16; ++ks) {
        uint32_t vb[2][4];
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          const int vr = 16 * ks + ri + (mi & 1) * 8;
          const int vc = (32 * wid + 16 * np) / 8 + (mi >> 1);
          ldsm_x4_t(vb[np][0], vb[np][1], vb[np][2], vb[np][3], kv_u + swz1k(vr, vc));
#pragma unroll
          for (int k = 0; k < 4; ++k) vb[np][k] = bf16x2_to_f16x2(vb[np][k]);
        }
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
          uint32_t a0, a1, a2, a3;
          const int ph = 16 * mt + ri + (mi & 1) * 8;
          ldsm_x4(a0, a1, a2, a3, ps_u + swzp(ph, 2 * ks + (mi >> 1)));
#pragma unroll
          for (int nt = 0; nt < 4; ++nt)
            mma_f16(acc_o[mt][nt], a0, a1, a2, a3, vb[nt >> 1][2 * (nt & 1)], vb[nt >> 1][2 * (nt & 1) + 1]);
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  if (n_split == 1) {
    // ---- finish the row: sink in the denominator, normalise, inverse RoPE
    // per-head statistics from the QK warps (replicated across the 4 row blocks)
    if ((wid >> 2) == 0 && c == 0) {
      sm.red_max[0][hq + g] = m_run[0];
      sm.red_max[0][hq + g + 8] = m_run[1];
      sm.red_sum[0][hq + g] = l_run[0];
      sm.red_sum[0][hq + g + 8] = l_run[1];
    }
    __syncthreads();
    if (tid < kHeads) {
      const float m = sm.red_max[0][tid], l = sm.red_sum[0][tid], sk = __ldg(p.sink + tid);
      const float M = fmaxf(m, sk);
      const float em = m == -INFINITY ? 0.f : __expf(m - M);
      const float den = l * em + __expf(sk - M);
      sm.alpha[tid] = em / den;  // multiplies the unnormalised output
      if (p.sink_mass) p.sink_mass[(size_t)row * kHeads + tid] = __expf(sk - M) / den;
    }
    __syncthreads();
    rope_table(sm.cs, p, qp, -1.f);
    __syncthreads();
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int h = 16 * mt + g + 8 * hh;
        const float f = sm.alpha[h];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const int d = 32 * wid + 8 * nt + 2 * c;
          float x = acc_o[mt][nt][2 * hh] * f, y = acc_o[mt][nt][2 * hh + 1] * f;
          if (d >= kHeadDim - kRopeDim) {
            const int i = (d - (kHeadDim - kRopeDim)) >> 1;
            const float cs = sm.cs[i], sn = sm.cs[32 + i];
            const float xr = x * cs - y * sn, yr = x * sn + y * cs;
            x = xr;
            y = yr;
          }
          *reinterpret_cast<float2*>(p.out + ((size_t)row * kHeads + h) * kHeadDim + d) = make_float2(x, y);
        }
      }
    return;
  }
  // ---- partial results of this split
  float* po = p.part_o + ((size_t)row * n_split + split) * kHeads * kHeadDim;
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int h = 16 * mt + g + 8 * hh;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int d = 32 * wid + 8 * nt + 2 * c;
        *reinterpret_cast<float2*>(po + (size_t)h * kHeadDim + d) =
            make_float2(acc_o[mt][nt][2 * hh], acc_o[mt][nt][2 * hh + 1]);
      }
    }
  if ((wid >> 2) == 0 && c == 0) {
    float* pm = p.part_ml + ((size_t)row * n_split + split) * kHeads * 2;
    pm[2 * (hq + g)] = m_run[0];
    pm[2 * (hq + g) + 1] = l_run[0];
    pm[2 * (hq + g + 8)] = m_run[1];
    pm[2 * (hq + g + 8) + 1] = l_run[1];
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
  cudaError_t e = cudaFuncSetAttribute(attn_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kAttnSmemBytes);
  if (e != cudaSuccess) return e;
  attn_split_kernel<<<dim3(n_split, p.n_rows), kAttnThreads, kAttnSmemBytes, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess || n_split == 1) return e;
  attn_combine_kernel<<<dim3(p.n_rows, kHeads / 4), 128, 0, stream>>>(p, n_split);
  return cudaGetLastError();
}

}  // namespace csa2
