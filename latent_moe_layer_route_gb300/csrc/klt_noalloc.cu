// Allocation-free routing + permutation entry point.
//
// Some callers cannot allocate device memory at the point where they route tokens: code
// that runs inside another framework's memory pool and may not call cudaMalloc, serving
// loops that pin every allocation at start-up so nothing can fail or stall mid-request,
// and embedded runtimes whose allocator is not reachable from the routing call.  For them
// klt_route_noalloc runs the same routing and permutation kernels as klt_forward without a
// handle and without any allocation: the per-block histogram and the other internal
// buffers live in one fixed-size array in device global memory, declared below, that every
// GPU loading this library holds until the process exits.
//
// The array is shared by every call in the process on a given device, so two calls whose
// kernels overlap on the GPU (different streams without ordering) race on it; calls must
// be ordered.  Every byte a call reads from it is written earlier in the same call, so no
// state carries over and nothing needs clearing between calls.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/klt.h"
#include "klt_internal.h"

namespace {

// Scratch layout (ints): per-block expert histogram [max blocks][MAX_E], tile offsets
// [MAX_E + 1] (written by the permutation, unused here), permuted routing weights
// [max pairs] (same).
constexpr int kMaxBlocks = (KLT_NOALLOC_MAX_PAIRS + klt::PERM_BLOCK - 1) / klt::PERM_BLOCK;
constexpr int kHistInts = kMaxBlocks * klt::MAX_E;
constexpr int kTileOffInts = klt::MAX_E + 1 + 3;  // padded to keep the next part aligned
constexpr int kScratchInts = kHistInts + kTileOffInts + KLT_NOALLOC_MAX_PAIRS;

static __device__ __align__(256) int g_route_scratch[kScratchInts];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array for the current device, resolved once per device.
// In host code the array's name is only a host-side stand-in, never a device address.
int scratch_for_current_device(int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return KLT_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_route_scratch) != cudaSuccess || !ptr)
      return KLT_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<int*>(ptr);
  }
  *out = g_scratch_ptr[dev];
  return KLT_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int klt_route_noalloc(const float* logits, int32_t M, int32_t E, int32_t topk,
                                 int32_t* ids, float* weights, int32_t* cnt, int32_t* off,
                                 int32_t* gidx, int32_t* slot, int32_t* pos, void* stream) {
  if (M < 0 || E < 1 || topk < 1) return KLT_ERR_INVALID_ARG;
  if (E > klt::MAX_E || topk > E || topk > klt::MAX_TOPK) return KLT_ERR_UNSUPPORTED;
  if (static_cast<long long>(M) * topk > KLT_NOALLOC_MAX_PAIRS) return KLT_ERR_TOO_LARGE;
  if (M == 0) return KLT_OK;
  const void* ptrs[] = {logits, ids, weights, cnt, off, gidx, slot, pos};
  for (const void* q : ptrs)
    if (!q) return KLT_ERR_INVALID_ARG;
  for (const void* q : ptrs)
    if (!aligned16(q)) return KLT_ERR_ALIGN;
  int* scratch = nullptr;
  int rc = scratch_for_current_device(&scratch);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int Mk = M * topk;
  const int nblocks = (Mk + klt::PERM_BLOCK - 1) / klt::PERM_BLOCK;

  klt::RouteParams rp = {};
  rp.logits = logits;
  rp.ids = ids;
  rp.wts = weights;
  rp.nsched = 0;
  rp.M = M;
  rp.E = E;
  rp.k = topk;
  rp.L = 0;  // routing only: no latent groups to quantise
  if (klt::launch_route(rp, s, false) != cudaSuccess) return KLT_ERR_CUDA;

  klt::PermParams pp = {};
  pp.ids = ids;
  pp.hist = scratch;
  pp.cnt = cnt;
  pp.off = off;
  pp.tile_off = scratch + kHistInts;
  pp.gidx = gidx;
  pp.slot = slot;
  pp.pos = pos;
  pp.wts = weights;
  pp.wperm = reinterpret_cast<float*>(scratch + kHistInts + kTileOffInts);
  pp.M = M;
  pp.E = E;
  pp.k = topk;
  pp.L = 0;
  pp.cap = Mk;
  pp.bn = 16;
  pp.nblocks = nblocks;
  if (nblocks > 1 && klt::launch_perm_hist(pp, s, false) != cudaSuccess) return KLT_ERR_CUDA;
  if (klt::launch_perm_scatter(pp, s, false) != cudaSuccess) return KLT_ERR_CUDA;
  return KLT_OK;
}
