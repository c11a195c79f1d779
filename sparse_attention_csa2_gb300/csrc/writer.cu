// Cache writer: records into a main-KV cache (FP4: E2M1 codes with one E4M3 scale per 16 or
// 32 channels; or bf16) or a sliding-window cache (FP8 rows with one fp32 scale), each record's rotary
// coordinates turned by its position first (the course's FP4 lesson, section 4: the cache is
// quantized after RoPE; "DeepSeek-V4.1-Flash explained", section 7: E2M1 with one E4M3
// scale per 16 channels; the local cache stays FP8).
//
// One warp per record, lane l holding dims 16l .. 16l+15 (one FP4 group of 16; lane pairs
// form a group of 32).  Every decision is taken in IEEE float32: the divisions are
// correctly rounded (__fdiv_rn), the rotation's products and sums are separate roundings
// (no fused multiply-add), and cos and sin come from double precision, rounded to float.
#include "common.cuh"
#include "kernels.h"

namespace csa2 {
namespace {

constexpr int kWriteWarps = 8;

__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {  // lo in the low byte
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {  // lo in the low nibble
  uint32_t r;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u32.u8 %0, t;\n}\n"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  const uint32_t h = e4m3x2_to_f16x2((uint16_t)(code & 0xffu));
  return __half2float(__ushort_as_half((unsigned short)(h & 0xffffu)));
}

// Sequence compressor: one warp per entry, lane l holding channels 16l .. 16l+15; per
// channel a softmax over the entry's `ratio` gate logits weighs its tokens' values (the
// encoder's banks pool consecutive tokens with learned channel-wise softmax gates, course,
// "How CSA2 compresses, shares, and selects attention memory").
template <bool F32>
__device__ __forceinline__ void load16(const void* base, long long row, int lane, float (&v)[16]) {
  if (F32) {
    const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(base) + row * kHeadDim + 16 * lane);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 f = __ldg(src + q);
      v[4 * q] = f.x, v[4 * q + 1] = f.y, v[4 * q + 2] = f.z, v[4 * q + 3] = f.w;
    }
  } else {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + row * kHeadDim + 16 * lane);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint4 u = __ldg(src + q);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        v[8 * q + 2 * k] = __uint_as_float(w[k] << 16);
        v[8 * q + 2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
      }
    }
  }
}

__global__ void __launch_bounds__(kWriteWarps * 32) write_records_kernel(const WriteParams p) {
  const int lane = threadIdx.x & 31;
  const long long r = (long long)blockIdx.x * kWriteWarps + (threadIdx.x >> 5);
  if (r >= p.n_rows) return;
  const long long dst = p.dst_row[r];
  if (dst < 0 || dst >= p.cache_rows) {
    if (lane == 0 && p.dev_status) atomicExch(p.dev_status, (int)CSA2_EDEVICE_INDEX);
    return;
  }
  // the lane's 16 values
  float v[16];
  if (p.x_f32)
    load16<true>(p.x, r, lane, v);
  else
    load16<false>(p.x, r, lane, v);
  // rotation: lane i forms cos and sin of pair i (angle pos * theta^(-2i/64), reduced modulo
  // 2 pi in double with a two-part 2 pi, then double sincos of |r| <= pi, rounded to float);
  // lanes 28..31 hold the pairs (448 + 2i, 449 + 2i), 8 each, and fetch theirs
  if (p.pos != nullptr) {
    const double a = (double)p.pos[r] * p.inv_freq[lane];
    const double kq = rint(a * 0.15915494309189535);  // 1 / (2 pi)
    double rr = fma(-kq, 6.283185307179586, a);
    rr = fma(-kq, 2.4492935982947064e-16, rr);
    double sd, cd;
    sincos(rr, &sd, &cd);
    const float cl = (float)cd, sl = (float)sd;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int src = 8 * (lane & 3) + k;  // lanes 28..31: pairs 8 (lane - 28) + k
      const float c = __shfl_sync(0xffffffffu, cl, src), s = __shfl_sync(0xffffffffu, sl, src);
      if (lane >= 28) {
        const float x = v[2 * k], y = v[2 * k + 1];
        v[2 * k] = __fsub_rn(__fmul_rn(x, c), __fmul_rn(y, s));
        v[2 * k + 1] = __fadd_rn(__fmul_rn(x, s), __fmul_rn(y, c));
      }
    }
  }
  if (p.out_dtype == CSA2_BF16) {  // rotated record in bf16, rounded to nearest even
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
      w[k] = *reinterpret_cast<const uint32_t*>(&h);
    }
    uint4* row = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.codes) + dst * kHeadDim + 16 * lane);
    row[0] = make_uint4(w[0], w[1], w[2], w[3]);
    row[1] = make_uint4(w[4], w[5], w[6], w[7]);
    return;
  }
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(v[k]));

  if (p.out_dtype == CSA2_FP8_E4M3_ROWSCALE) {
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t b01 = f32x2_to_e4m3x2(__fdiv_rn(v[4 * k], scale), __fdiv_rn(v[4 * k + 1], scale));
      const uint32_t b23 = f32x2_to_e4m3x2(__fdiv_rn(v[4 * k + 2], scale), __fdiv_rn(v[4 * k + 3], scale));
      w[k] = (b01 & 0xffffu) | (b23 << 16);
    }
    uint8_t* codes = static_cast<uint8_t*>(p.codes) + dst * kHeadDim;
    *reinterpret_cast<uint4*>(codes + 16 * lane) = make_uint4(w[0], w[1], w[2], w[3]);
    if (lane == 0) static_cast<float*>(p.scales)[dst] = scale;
    return;
  }
  // FP4: the group's scale is the smallest E4M3 value at or above amax / 6
  const bool g32 = p.out_dtype == CSA2_FP4_E2M1_G32;
  if (g32) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  const float s = __fdiv_rn(amax, 6.f);
  uint32_t code = f32x2_to_e4m3x2(s, 0.f) & 0xffu;  // nearest, saturating at 448
  if (e4m3_value(code) < s && code < 0x7eu) ++code;  // positive codes ascend with their value
  const float scale = e4m3_value(code);
  uint32_t packed[2] = {0u, 0u};
  if (scale > 0.f) {
#pragma unroll
    for (int k = 0; k < 8; ++k)
      packed[k >> 2] |= f32x2_to_e2m1x2(__fdiv_rn(v[2 * k], scale), __fdiv_rn(v[2 * k + 1], scale)) << (8 * (k & 3));
  }
  uint8_t* codes = static_cast<uint8_t*>(p.codes) + dst * (kHeadDim / 2);
  *reinterpret_cast<uint2*>(codes + 8 * lane) = make_uint2(packed[0], packed[1]);
  uint8_t* sc = static_cast<uint8_t*>(p.scales);
  if (!g32) sc[dst * (kHeadDim / 16) + lane] = (uint8_t)code;
  else if ((lane & 1) == 0) sc[dst * (kHeadDim / 32) + lane / 2] = (uint8_t)code;
}

template <bool F32>
__global__ void __launch_bounds__(kWriteWarps * 32)
    compress_kernel(long long n_entries, int ratio, const void* kv, const void* gate, float* out) {
  const int lane = threadIdx.x & 31;
  const long long e = (long long)blockIdx.x * kWriteWarps + (threadIdx.x >> 5);
  if (e >= n_entries) return;
  float m[16], den[16], num[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) m[k] = -INFINITY, den[k] = 0.f, num[k] = 0.f;
  // online softmax over the entry's tokens, channel by channel
#pragma unroll 1
  for (int j = 0; j < ratio; ++j) {
    float g[16], x[16];
    load16<F32>(gate, e * ratio + j, lane, g);
    load16<F32>(kv, e * ratio + j, lane, x);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float mn = fmaxf(m[k], g[k]);
      const float a = __expf(m[k] - mn), b = __expf(g[k] - mn);
      den[k] = den[k] * a + b;
      num[k] = num[k] * a + b * x[k];
      m[k] = mn;
    }
  }
  float4* dst = reinterpret_cast<float4*>(out + e * kHeadDim + 16 * lane);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    dst[q] = make_float4(num[4 * q] / den[4 * q], num[4 * q + 1] / den[4 * q + 1], num[4 * q + 2] / den[4 * q + 2],
                         num[4 * q + 3] / den[4 * q + 3]);
}

// MXFP4 rows (64 code bytes + 4 UE8M0 exponents per 128-element record) -> their bf16 values:
// one thread per block of 32 elements (16 code bytes, one exponent); every E2M1 level times a
// power of two 2^(e - 127), e < 255, is a bf16 value (normal or subnormal), so the expansion
// is exact; e = 255 (the OCP NaN scale) gives NaN.
__global__ void __launch_bounds__(256) expand_mxfp4_kernel(long long n_blocks, const uint8_t* codes,
                                                            const uint8_t* exps, uint16_t* out) {
  const long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= n_blocks) return;
  const uint4 c = __ldg(reinterpret_cast<const uint4*>(codes) + b);
  const uint32_t e = __ldg(exps + b);
  const float scale = e == 255u ? __uint_as_float(0x7fc00000u)
                      : e == 0u ? __uint_as_float(0x00400000u)  // 2^-127, a subnormal
                                : __uint_as_float(e << 23);
  const uint32_t w4[4] = {c.x, c.y, c.z, c.w};
  uint32_t o[16];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int byte = 0; byte < 4; ++byte) {
      const uint32_t h = e2m1x2_to_f16x2((w4[k] >> (8 * byte)) & 0xffu);
      const float lo = __half2float(__ushort_as_half((unsigned short)(h & 0xffffu))) * scale;
      const float hi = __half2float(__ushort_as_half((unsigned short)(h >> 16))) * scale;
      const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
      o[4 * k + byte] = *reinterpret_cast<const uint32_t*>(&v);
    }
  }
  uint4* dst = reinterpret_cast<uint4*>(out + b * 32);
#pragma unroll
  for (int q = 0; q < 4; ++q) dst[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
}

}  // namespace

cudaError_t launch_expand_mxfp4(long long n_records, const void* codes, const void* exps, void* out,
                                cudaStream_t stream) {
  if (n_records == 0) return cudaSuccess;
  const long long n_blocks = n_records * 4;
  expand_mxfp4_kernel<<<(unsigned)((n_blocks + 255) / 256), 256, 0, stream>>>(
      n_blocks, static_cast<const uint8_t*>(codes), static_cast<const uint8_t*>(exps), static_cast<uint16_t*>(out));
  return cudaGetLastError();
}

cudaError_t launch_compress(long long n_entries, int ratio, const void* kv, const void* gate, bool x_f32, float* out,
                            cudaStream_t stream) {
  if (n_entries == 0) return cudaSuccess;
  const long long blocks = (n_entries + kWriteWarps - 1) / kWriteWarps;
  if (x_f32)
    compress_kernel<true><<<(unsigned)blocks, kWriteWarps * 32, 0, stream>>>(n_entries, ratio, kv, gate, out);
  else
    compress_kernel<false><<<(unsigned)blocks, kWriteWarps * 32, 0, stream>>>(n_entries, ratio, kv, gate, out);
  return cudaGetLastError();
}

cudaError_t launch_write_records(const WriteParams& p, cudaStream_t stream) {
  if (p.n_rows == 0) return cudaSuccess;
  const long long blocks = (p.n_rows + kWriteWarps - 1) / kWriteWarps;
  write_records_kernel<<<(unsigned)blocks, kWriteWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace csa2
