// Projections on either side of CSA2 attention ("DeepSeek V4.1-Flash. Every layer, connected",
// "The query and output paths": a low-rank query projection and a grouped output projection;
// "DeepSeek V4 Inside": the Flash config's query rank 1024, RMSNorm on the query head, the 64
// heads' outputs through a grouped W_O with 8 groups).
//
// One kernel computes out[t, f] = sum_k W[f, k] x[t, k] on the tensor cores, the weights as the
// A operand (128 features per block: the MMA's M) and the tokens as B (a tile of bn tokens: the
// MMA's N), so that at decode, with few tokens, each weight is read from HBM once.  Warp 0
// issues the TMA loads (the first stages' weight tiles before it waits for the preceding
// kernel, which the weights do not depend on), warp 1 the MMAs into tensor memory, warps 2..5
// run the epilogue, one accumulator lane (feature) per thread.  Epilogues:
//   plain  bf16 store; grouped, group g reads its own columns of B (its heads) and writes its
//          own columns of out;
//   down   bf16 store of acc * g_q[f], and per token the sum of acc^2 over the block's
//          features (the RMSNorm of the query's low-rank vector is finished by the next
//          launch);
//   up     acc times the token's low-rank RMSNorm factor, then RMSNorm over each head's 512
//          features: the four blocks of a head form a cluster and exchange their per-token
//          sums of squares through distributed shared memory; then the head gain.
// The output tile is staged in the (then idle) pipeline buffers as token rows and written with
// 16-byte stores.  With ks > 1 the K range is split over a cluster of ks blocks; each block
// stages its fp32 accumulator, and block r reads rows [r R, r R + R) (R = 128 / ks) of every
// block's staged tile, adds them in rank order and finishes those rows.
#include "common.cuh"
#include "kernels.h"
#include "tc05.cuh"

namespace csa2 {
namespace {

constexpr int kProjThreads = 192;
constexpr int kATile = 128 * 128;  // 128 weight rows x 64 bf16 (128 bytes)

struct ProjShared {
  uint64_t full[kProjMaxStages];
  uint64_t empty[kProjMaxStages];
  uint64_t done;
  uint32_t tmem_base;
  int timeout;
  int issued, consumed;
  alignas(16) float tok[256];  // up: per-token factor (read as float4)
  float red[4][256];  // per epilogue warp and token: sums of squares over the warp's 32 features
  float xch[4][256];  // up: per cluster rank and token: that block's sum of squares
  float gain[128];    // the gain of each of the tile's features (1 without gains)
};

__device__ __forceinline__ uint8_t* align1024_proj(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}
__device__ __forceinline__ void proj_timeout(int* flag, int32_t* dev_status) {
  *flag = 1;
  if (dev_status != nullptr) atomicExch(dev_status, (int)CSA2_ETIMEOUT);
}
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;\n" ::: "memory"); }
__device__ __forceinline__ void cluster_st_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;\n" ::"r"(addr), "f"(v) : "memory");
}

// A load from another block's shared memory that the compiler may schedule freely (the data
// is ordered by the cluster barrier before it).
__device__ __forceinline__ uint4 cluster_ld_v4_nv(uint32_t addr) {
  uint4 v;
  asm("ld.shared::cluster.v4.u32 {%0,%1,%2,%3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// 32 values per lane -> lane l returns the warp's sum of value l (a butterfly: at each step a
// lane keeps half of its values and adds its partner's half; 31 shuffles).
__device__ __forceinline__ float warp_sum_scatter32(float (&a)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float give = upper ? a[i] : a[i + w];
      const float keep = upper ? a[i + w] : a[i];
      a[i] = keep + __shfl_xor_sync(0xffffffffu, give, w);
    }
  }
  return a[0];
}

__global__ void __launch_bounds__(kProjThreads, 1)
    proj_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const ProjParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = align1024_proj(smem_raw);
  const int stage_bytes = kATile + p.bn * 128;
  ProjShared& sh = *reinterpret_cast<ProjShared*>(ring + p.stages * stage_bytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.z;
  const int m_tile = blockIdx.x / p.ks, split = blockIdx.x % p.ks;
  const int n0 = blockIdx.y * p.bn;
  const int s0 = (int)((long long)p.k_steps * split / p.ks);
  const int n_steps = (int)((long long)p.k_steps * (split + 1) / p.ks) - s0;
  const int a_row = g * p.a_rows_per_group + m_tile * 128;
  const int b_col = g * p.b_cols_per_group;
  const uint32_t tmem_cols = (uint32_t)p.bn;

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      tc05::mbar_init(&sh.full[s], 1);
      tc05::mbar_init(&sh.empty[s], 1);
    }
    tc05::mbar_init(&sh.done, 1);
    sh.timeout = 0;
    sh.issued = sh.consumed = 0;
    tc05::fence_barrier_init();
  }
  if (warp == 1) tc05::tmem_alloc(&sh.tmem_base, tmem_cols);
  tc05::fence_before();
  __syncthreads();
  tc05::fence_after();
  const uint32_t tmem = sh.tmem_base;
  // the next kernel may start: this block already holds its tensor memory
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      const int pre = min(n_steps, p.stages);
      for (int i = 0; i < pre; ++i) {
        tc05::mbar_expect_tx(&sh.full[i], stage_bytes);
        tc05::tma_load_2d(ring + i * stage_bytes, &tmA, (s0 + i) * 64, a_row, &sh.full[i]);
      }
      asm volatile("griddepcontrol.wait;\n" ::: "memory");  // B is the preceding kernel's output
      bool ok = true;
      for (int i = 0; i < n_steps; ++i) {
        const int s = i % p.stages;
        uint8_t* st = ring + s * stage_bytes;
        if (i >= p.stages) {
          if (!tc05::mbar_wait(&sh.empty[s], ((i / p.stages) & 1) ^ 1)) {
            ok = false;
            break;
          }
          tc05::mbar_expect_tx(&sh.full[s], stage_bytes);
          tc05::tma_load_2d(st, &tmA, (s0 + i) * 64, a_row, &sh.full[s]);
        }
        tc05::tma_load_2d(st + kATile, &tmB, b_col + (s0 + i) * 64, n0, &sh.full[s]);
        sh.issued = i + 1;
      }
      if (!ok) proj_timeout(&sh.timeout, p.dev_status);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc05::idesc_bf16(128, p.bn);
      bool ok = true;
      for (int i = 0; i < n_steps; ++i) {
        const int s = i % p.stages;
        if (!tc05::mbar_wait(&sh.full[s], (i / p.stages) & 1)) {
          ok = false;
          break;
        }
        tc05::fence_after();
        const uint32_t a_u = smem_u32(ring + s * stage_bytes), b_u = a_u + kATile;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc05::mma_bf16(tmem, tc05::sw128_desc(a_u + kk * 32), tc05::sw128_desc(b_u + kk * 32), idesc,
                         (i | kk) != 0);
        tc05::mma_commit(&sh.empty[s]);
        sh.consumed = i + 1;
      }
      if (ok)
        tc05::mma_commit(&sh.done);
      else
        proj_timeout(&sh.timeout, p.dev_status);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue: wait
    const int et = tid - 64;
    if (p.mode == kProjUp) {
      // the token's low-rank RMSNorm factor, from the down-projection's partial sums
      asm volatile("griddepcontrol.wait;\n" ::: "memory");
      for (int j = et; j < p.bn; j += 128) {
        const int t = n0 + j;
        float s = 0.f;
        if (t < p.n_tok)
          for (int i = 0; i < p.ss_tiles; ++i) s += p.ss[(size_t)i * p.n_tok + t];
        sh.tok[j] = rsqrtf(s * p.inv_rank + p.eps);
      }
    }
    // the tile's gains, read while the MMAs run
    {
      const int f = m_tile * 128 + et;
      sh.gain[et] = p.gain == nullptr || p.mode == kProjPlain ? 1.f
                    : __ldg(p.gain + (p.mode == kProjUp ? (f & (kHeadDim - 1)) : f));
    }
    epi_sync();  // the gains are read by other threads than their writers
    if (!tc05::mbar_wait(&sh.done, 0) && lane == 0) proj_timeout(&sh.timeout, p.dev_status);
    tc05::fence_after();
  }

  __syncthreads();
  const bool clustered = p.ks > 1 || p.mode == kProjUp;
  const uint32_t rank = clustered ? cluster_rank() : 0u;
  // every block of the cluster has its accumulator, so every pipeline buffer is idle
  if (clustered) cluster_sync();

  const int quarter = warp & 3;                 // TMEM lanes 32 * quarter .. + 31
  const int row = 32 * quarter + lane;          // this thread's feature within the tile
  const int et = tid - 64;
  const bool epi = warp >= 2;
  const uint32_t t_lane = tmem + ((uint32_t)(32 * quarter) << 16);
  const int n_chunks = p.bn / 32;
  __nv_bfloat16* const outg = static_cast<__nv_bfloat16*>(p.out) + (size_t)g * p.out_cols_per_group + m_tile * 128;

  if (p.ks > 1) {
    // ---------------------------------------------------------------- split K
    // every block stages its accumulator as token rows, [bn][128 + 4] fp32; block r then reads
    // rows [r R, r R + R) (R = 128 / ks) of every block's staged tile through distributed shared
    // memory, adds them in rank order and finishes those features, 8 per thread and token
    constexpr int kLd = 128 + 4;
    float* stg = reinterpret_cast<float*>(ring);
    if (epi) {
      for (int c = 0; c < n_chunks; ++c) {
        uint32_t v[32];
        tc05::tmem_ld32(t_lane + 32 * c, v);
        tc05::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) stg[(32 * c + j) * kLd + row] = __uint_as_float(v[j]);
      }
    }
    cluster_sync();  // every block's tile is staged
    if (epi) {
      const int R = 128 / p.ks, n_oct = R / 8, f0 = (int)rank * R;
      // bn * n_oct is a multiple of 64, so whole warps take part in every iteration
      for (int i = et; i < p.bn * n_oct; i += 128) {
        const int t = i / n_oct, o = i - t * n_oct, tok = n0 + t;
        const uint32_t off = (uint32_t)(t * kLd + f0 + 8 * o) * 4u;
        // all of the (at most 8) blocks' pieces are requested before any is added, so the
        // remote loads overlap
        uint4 lo[8], hi[8];
#pragma unroll
        for (int src = 0; src < 8; ++src) {
          if (src < p.ks) {
            const uint32_t at = cluster_map(stg, (uint32_t)src) + off;
            lo[src] = cluster_ld_v4_nv(at);
            hi[src] = cluster_ld_v4_nv(at + 16u);
          }
        }
        float y[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int src = 0; src < 8; ++src) {
          if (src < p.ks) {
            y[0] += __uint_as_float(lo[src].x), y[1] += __uint_as_float(lo[src].y);
            y[2] += __uint_as_float(lo[src].z), y[3] += __uint_as_float(lo[src].w);
            y[4] += __uint_as_float(hi[src].x), y[5] += __uint_as_float(hi[src].y);
            y[6] += __uint_as_float(hi[src].z), y[7] += __uint_as_float(hi[src].w);
          }
        }
        float ss = 0.f;
        if (p.mode == kProjDown) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            ss = fmaf(y[k], y[k], ss);
            y[k] *= sh.gain[f0 + 8 * o + k];
          }
          for (int w = n_oct >> 1; w >= 1; w >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, w);
        }
        if (tok < p.n_tok) {
          uint4 w;
          w.x = pack_bf16x2(y[0], y[1]), w.y = pack_bf16x2(y[2], y[3]);
          w.z = pack_bf16x2(y[4], y[5]), w.w = pack_bf16x2(y[6], y[7]);
          *reinterpret_cast<uint4*>(outg + (size_t)tok * p.out_ld + f0 + 8 * o) = w;
          if (p.mode == kProjDown && o == 0) p.ss[(size_t)(m_tile * p.ks + (int)rank) * p.n_tok + tok] = ss;
        }
      }
    }
    cluster_sync();  // no block leaves while the others read its staged tile
  } else {
    // ---------------------------------------------------------------- whole K in this block
    if (epi && p.mode == kProjUp) {
      // per token, this block's sum of squares over its 128 features, sent to the cluster
      for (int c = 0; c < n_chunks; ++c) {
        uint32_t v[32];
        tc05::tmem_ld32(t_lane + 32 * c, v);
        float a[32];
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          const float4 q = *reinterpret_cast<const float4*>(&sh.tok[32 * c + j]);
          a[j] = q.x, a[j + 1] = q.y, a[j + 2] = q.z, a[j + 3] = q.w;
        }
        tc05::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float x = __uint_as_float(v[j]) * a[j];
          a[j] = x * x;
        }
        sh.red[quarter][32 * c + lane] = warp_sum_scatter32(a, lane);
      }
      epi_sync();
      for (int j = et; j < p.bn; j += 128) {
        const float part = (sh.red[0][j] + sh.red[1][j]) + (sh.red[2][j] + sh.red[3][j]);
        for (uint32_t r = 0; r < 4; ++r) cluster_st_f32(cluster_map(&sh.xch[rank][j], r), part);
      }
    }
    if (clustered) cluster_sync();  // the head sums are in place
    if (epi) {
      if (p.mode == kProjUp) {
        for (int j = et; j < p.bn; j += 128) {
          const float tot = (sh.xch[0][j] + sh.xch[1][j]) + (sh.xch[2][j] + sh.xch[3][j]);
          sh.tok[j] *= rsqrtf(tot * (1.f / (float)kHeadDim) + p.eps);
        }
        epi_sync();
      }
      // the tile's output goes through shared memory, [bn tokens][128 features] bf16 rows
      // (padded), and out to global memory in 16-byte pieces
      constexpr int kSld = 128 + 8;
      __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(ring);
      const float gain = sh.gain[row];
      for (int c = 0; c < n_chunks; ++c) {
        uint32_t v[32];
        tc05::tmem_ld32(t_lane + 32 * c, v);
        // per-token factors in registers first: the staging stores below could alias them
        float fac[32];
        if (p.mode == kProjUp) {
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 q = *reinterpret_cast<const float4*>(&sh.tok[32 * c + j]);
            fac[j] = q.x * gain, fac[j + 1] = q.y * gain, fac[j + 2] = q.z * gain, fac[j + 3] = q.w * gain;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) fac[j] = p.mode == kProjDown ? gain : 1.f;
        }
        tc05::tmem_ld_wait();
        float acc[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          acc[j] = __uint_as_float(v[j]);
          stage[(32 * c + j) * kSld + row] = __float2bfloat16_rn(acc[j] * fac[j]);
        }
        if (p.mode == kProjDown) {
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[j] *= acc[j];
          sh.red[quarter][32 * c + lane] = warp_sum_scatter32(acc, lane);
        }
      }
      epi_sync();
      for (int i = et; i < p.bn * 16; i += 128) {
        const int t = i >> 4, pc = i & 15;
        if (n0 + t < p.n_tok)
          *reinterpret_cast<uint4*>(outg + (size_t)(n0 + t) * p.out_ld + pc * 8) =
              *reinterpret_cast<const uint4*>(stage + t * kSld + pc * 8);
      }
      if (p.mode == kProjDown) {
        for (int j = et; j < p.bn; j += 128) {
          const int t = n0 + j;
          if (t < p.n_tok)
            p.ss[(size_t)m_tile * p.n_tok + t] = (sh.red[0][j] + sh.red[1][j]) + (sh.red[2][j] + sh.red[3][j]);
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (sh.timeout && tid == 0) {
    for (int i = sh.consumed; i < sh.issued; ++i) tc05::mbar_wait(&sh.full[i % p.stages], (i / p.stages) & 1);
    if (sh.consumed > 0) {
      const int i = sh.consumed - 1;
      tc05::mbar_wait(&sh.empty[i % p.stages], (i / p.stages) & 1);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc05::fence_after();
    tc05::tmem_dealloc(tmem, tmem_cols);
  }
}

}  // namespace

size_t proj_epilogue_bytes(int bn, int ks) {
  // the staged tile: fp32 accumulators with a K split, else the bf16 output
  return ks > 1 ? (size_t)bn * (128 + 4) * 4 : (size_t)bn * (128 + 8) * 2;
}

size_t proj_smem_bytes(int bn, int stages) {
  return 1024 + (size_t)stages * (kATile + (size_t)bn * 128) + sizeof(ProjShared);
}

cudaError_t launch_proj(const CUtensorMap& tmA, const CUtensorMap& tmB, const ProjParams& p, int groups,
                        cudaStream_t stream) {
  if (p.stages < 1 || p.stages > kProjMaxStages) return cudaErrorInvalidValue;
  const size_t smem = proj_smem_bytes(p.bn, p.stages);
  if (smem > 227 * 1024 || (size_t)p.stages * (kATile + (size_t)p.bn * 128) < proj_epilogue_bytes(p.bn, p.ks))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // may start before the preceding kernel in the stream has finished (programmatic dependent
  // launch): it waits for it before reading its output
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n_attr = 1;
  const int cl = p.mode == kProjUp ? 4 : p.ks;
  if (cl > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cl;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n_attr = 2;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.m_tiles * p.ks, (p.n_tok + p.bn - 1) / p.bn, groups);
  cfg.blockDim = dim3(kProjThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = n_attr;
  return cudaLaunchKernelEx(&cfg, proj_kernel, tmA, tmB, p);
}

}  // namespace csa2
