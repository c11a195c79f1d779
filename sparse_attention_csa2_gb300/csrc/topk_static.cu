// csa2_topk_static: csa2_topk for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: code running where cudaMalloc is
// unavailable or forbidden (for example inside a stream that is being captured into a CUDA
// graph by a framework that owns all allocations, or a runtime with a fixed memory budget
// that admits no further allocations once it is up).  This entry point takes the scratch
// memory that csa2_topk would take from `workspace` out of an array that is part of the
// library image instead.  It allocates nothing.
//
// The array is a file-scope __device__ variable of CSA2_TOPK_STATIC_SCRATCH_BYTES bytes, so
// every GPU on which the library is loaded holds it until the process exits.  Host code
// cannot use the variable's name as a device address; the device address is obtained once
// per device with cudaGetSymbolAddress, with that device current, on the first call on it,
// and kept for the life of the process (a cudaDeviceReset is not noticed).
#include <mutex>

#include "../../include/csa2.h"
#include "kernels.h"

namespace csa2 {
namespace {

__device__ __align__(256) uint8_t g_topk_scratch[CSA2_TOPK_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_topk_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace
}  // namespace csa2

using namespace csa2;

extern "C" csa2_status csa2_topk_static(const csa2_topk_args* a, void* stream) {
  if (!a || a->n_rows < 0) return CSA2_EINVAL;
  if (a->n_rows == 0) return CSA2_OK;
  if (!a->scores || !a->n_valid || !a->idx || a->L < 1 || a->L > (1LL << 24)) return CSA2_EINVAL;
  if (a->K < 1 || a->K > CSA2_MAX_TOPK) return CSA2_EUNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The scratch address and the segment count are the current device's; kernels on a stream
  // of another device would be handed this device's address, so such a stream is refused.
  // The default stream handles always belong to the current device.
  if (s != nullptr && s != cudaStreamLegacy && s != cudaStreamPerThread) {
    int cur = 0, sdev = 0;
    if (cudaGetDevice(&cur) != cudaSuccess || cudaStreamGetDevice(s, &sdev) != cudaSuccess) return CSA2_ECUDA;
    if (sdev != cur) return CSA2_EINVAL;
  }
  const int n_seg = topk_segments(a->n_rows, a->L);
  FeedParams f{};
  f.n_rows = a->n_rows;
  f.K = a->K;
  f.scores = a->scores;
  f.scores_stride = a->L;
  f.n_valid = a->n_valid;
  f.valid_div = 1;
  f.cand = a->cand;
  f.cand_stride = a->L;
  if (n_seg == 1) {  // one pass, no scratch
    f.idx = a->idx;
    return launch_topk_feed(f, false, 1, s) == cudaSuccess ? CSA2_OK : CSA2_ECUDA;
  }
  // scratch: per-segment (key, position) lists, their counts and thresholds; all written by
  // the first kernel before the second reads them, so nothing needs clearing between calls
  const size_t lists = (size_t)a->n_rows * n_seg * a->K;
  const size_t need = 2 * up256(lists * 4) + 2 * up256((size_t)a->n_rows * n_seg * 4);
  if (need > (size_t)CSA2_TOPK_STATIC_SCRATCH_BYTES) return CSA2_EUNSUPPORTED;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return CSA2_ECUDA;
  uint8_t* p = static_cast<uint8_t*>(base);
  f.out_keys = reinterpret_cast<uint32_t*>(p);
  p += up256(lists * 4);
  f.out_pos = reinterpret_cast<int32_t*>(p);
  p += up256(lists * 4);
  f.out_cnt = reinterpret_cast<int32_t*>(p);
  p += up256((size_t)a->n_rows * n_seg * 4);
  f.out_thr = reinterpret_cast<uint32_t*>(p);
  if (launch_topk_feed(f, false, n_seg, s) != cudaSuccess) return CSA2_ECUDA;
  FeedParams m{};
  m.n_rows = a->n_rows;
  m.K = a->K;
  m.in_keys = f.out_keys;
  m.in_pos = f.out_pos;
  m.in_cnt = f.out_cnt;
  m.in_thr = f.out_thr;
  m.in_seg = n_seg;
  m.in_K = a->K;
  m.idx = a->idx;
  return launch_lists_merge(m, s) == cudaSuccess ? CSA2_OK : CSA2_ECUDA;
}
