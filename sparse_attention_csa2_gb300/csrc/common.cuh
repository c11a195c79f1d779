// Device helpers shared by the CSA2 kernels (sm_103a): PTX wrappers for cp.async,
// ldmatrix and warp-level MMA, order-preserving score keys, and block-wide scans.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "../../include/csa2.h"

namespace csa2 {

constexpr int kIdxHeads = CSA2_IDX_HEADS;  // 32
constexpr int kIdxDim = CSA2_IDX_DIM;      // 128
constexpr int kHeads = CSA2_HEADS;         // 64
constexpr int kHeadDim = CSA2_HEAD_DIM;    // 512
constexpr int kRopeDim = CSA2_ROPE_DIM;    // 64

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ----------------------------------------------------------------------------- score keys
// Order-preserving map of an fp32 score to a uint32 key: a larger score gives a larger key,
// and -0.0 maps to the key of +0.0.  Key 0 (the image of one negative-NaN pattern, never
// produced from finite inputs) marks "no candidate".
__device__ __forceinline__ uint32_t score_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}

// ----------------------------------------------------------------------------- cp.async
// 16-byte global->shared copy; when !valid nothing is read and the 16 bytes are zeroed.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)), "l"(gmem),
               "r"(valid ? 16 : 0)
               : "memory");
}
// 4-byte global->shared copy (4-byte aligned); when !valid the 4 bytes are zeroed.
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_u32(smem)), "l"(gmem),
               "r"(valid ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ----------------------------------------------------------------------------- ldmatrix
__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                        uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t& r0, uint32_t& r1, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                          uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// ----------------------------------------------------------------------------- warp MMA
// D(16x8, fp32) += A(16x16) * B(16x8); A row-major, B column-major fragments.
__device__ __forceinline__ void mma_bf16(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ----------------------------------------------------------------------------- conversions
// Two OCP E4M3 codes (low byte = first) -> two bf16 (exact: every E4M3 value is a bf16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint16_t v) {
  uint32_t h;
  asm("{\n .reg .b32 t;\n cvt.rn.f16x2.e4m3x2 t, %1;\n mov.b32 %0, t;\n}\n" : "=r"(h) : "h"(v));
  __half2 hh = *reinterpret_cast<__half2*>(&h);
  float2 f = __half22float2(hh);
  __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
  return *reinterpret_cast<uint32_t*>(&b);
}
// Two OCP E4M3 codes (low byte = first) -> two f16 (packed, exact: every E4M3 value is an f16
// value), by the hardware conversion.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t h;
  asm("{\n .reg .b32 t;\n cvt.rn.f16x2.e4m3x2 t, %1;\n mov.b32 %0, t;\n}\n" : "=r"(h) : "h"(v));
  return h;
}
// One byte of two E2M1 codes (low nibble first) -> two f16 (packed, exact), by the hardware
// conversion.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t h;
  asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}\n" : "=r"(h) : "r"(byte));
  return h;
}
// Two bf16 (packed) -> two fp16 (packed), round to nearest.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  float lo = __uint_as_float(v << 16);
  float hi = __uint_as_float(v & 0xffff0000u);
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// ----------------------------------------------------------------------------- block scans
// Exclusive prefix sum over the NT threads of a block; *total receives the block sum.
// `warp_tmp` is shared scratch of >= NT/32 ints.  Contains __syncthreads: call uniformly.
template <int NT>
__device__ __forceinline__ int block_excl_scan(int v, int* warp_tmp, int* total) {
  static_assert(NT % 32 == 0 && NT <= 1024, "block size");
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tmp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int t = lane < NW ? warp_tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < NW) warp_tmp[lane] = t;
  }
  __syncthreads();
  const int before = wid ? warp_tmp[wid - 1] : 0;
  *total = warp_tmp[NW - 1];
  __syncthreads();
  return before + x - v;
}

template <int NT>
__device__ __forceinline__ int block_sum(int v, int* warp_tmp) {
  int total;
  block_excl_scan<NT>(v, warp_tmp, &total);
  return total;
}

// Bit mask of the lanes below the calling one.
__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ----------------------------------------------------------------------------- clusters
// Rank of this block in its thread-block cluster, the cluster barrier (all threads of every
// block of the cluster; release / acquire order shared-memory accesses across the blocks),
// and loads / stores to another block's shared memory through its cluster address.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// The two halves of the cluster barrier: every thread of every block arrives once per phase
// and waits for the phase before it arrives again.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_map(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ uint4 cluster_ld_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0,%1,%2,%3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ int cluster_ld_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];\n" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void cluster_st_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1,%2,%3,%4};\n" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void cluster_st_s32(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;\n" ::"r"(addr), "r"(v) : "memory");
}

// ----------------------------------------------------------------------------- arrivals
// Counts one arrival (a finished part of a row) in `ctr` = tag << 32 | count, where another
// tag means an earlier call: the count restarts, so the counters need no clearing between
// calls.  Returns true for the arrival that completes the n parts.  Once a block of this call
// has installed the tag (one compare-and-swap), every other block counts with a single atomic
// add; the retries are bounded all the same.
__device__ __forceinline__ bool count_arrival(unsigned long long* ctr, uint32_t tag, int n, int32_t* dev_status) {
  unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(ctr);
  for (int tries = 0; tries < 64; ++tries) {
    if ((uint32_t)(cur >> 32) == tag) {
      const unsigned long long old = atomicAdd(ctr, 1ull);  // the tag stays for the whole call
      return (uint32_t)old + 1u == (uint32_t)n;
    }
    const unsigned long long prev = atomicCAS(ctr, cur, ((unsigned long long)tag << 32) | 1ull);
    if (prev == cur) return n == 1;
    cur = prev;
  }
  if (dev_status != nullptr) atomicExch(dev_status, (int)CSA2_ETIMEOUT);
  return false;
}

}  // namespace csa2
