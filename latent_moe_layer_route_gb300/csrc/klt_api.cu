// Host side of the latent-MoE tail C ABI: argument checks, owned weight copies, the
// workspace, TMA descriptor encoding and the per-forward launch chain
//
//   route_quant -> [perm_hist] -> perm_scatter -> perm_gather -> GEMM(shared L1 + routed L1)
//   -> GEMM(routed L2 + combine) -> norm -> GEMM(up-projection + shared L2 -> out)
//
// all on the caller's stream, chained with programmatic dependent launch.  The shared
// expert's down-projection is fused into the output GEMM as extra K blocks
// ([n | a_s] . [W_up | Ws2]^T), so the shared output is added to the up-projection in
// the fp32 accumulator and the result is rounded to bf16 once.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>

#include "../../include/klt.h"
#include "klt_internal.h"

using namespace klt;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// Row-major [rows, cols] matrix of `esize`-byte elements; box = box_cols x box_rows with
// box_cols * esize == 128 (one 128-byte swizzle row); out-of-range elements read as zero.
bool encode_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize,
               uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * static_cast<uint64_t>(esize)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esize), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kNumBN = 4;
constexpr int kBN[kNumBN] = {16, 32, 64, 128};
constexpr int kMaxSplitUnits = 3 * 160;  // split-K tiles*splits bound per task
constexpr int kMaxCounters = 8192;       // arrival counters per split launch
constexpr int kWideMinTokens = 17;  // token-major engine above the 16-token decode tile
constexpr int kDualMinTiles = 16;   // token-major units over two token tiles from 2048 tokens

}  // namespace

struct klt_handle {
  klt_dims d;
  uint32_t flags;
  int device;
  int num_sms;
  // owned weights
  uint8_t *w13, *w2;
  float *w13_s, *w2_s;
  __nv_bfloat16 *ws13, *ws2, *w_up, *gamma;
  // workspace
  int32_t *ids, *cnt, *off, *tile_off, *gidx, *slot, *pos, *hist;
  float *wts, *wperm, *zs, *zsT, *asT, *r, *ws;
  float* yw;  // deterministic combine: weighted output per (token, choice) slot, or null
  uint8_t *zq, *zq_perm, *aq;
  __nv_bfloat16 *n, *a_s, *zqb_perm, *aqb;
  int *split_cnt, *sched, *err;
  float* out_acc;  // token-major k-split output tiles (fp32, zero between forwards)
  int* out_cnt;    //   and their arrival counters
  int* dep_cnt;  // fused-launch dependency counters [routed tiles | l2 | norm tiles | shared]
  // Block-scaled layers (MXFP8, NVFP4_W4A4): weight scale tiles (512 bytes per 128-row
  // block and 4 scale bytes of a row, the tcgen05.cp layout), the latent input's scale
  // bytes, and the token scale tiles of the routed L1 and L2 units (per routed tile of 128
  // pairs); NVFP4_W4A4 also the weights' fp32 per-matrix scales [E]
  uint8_t *w13_sf, *w2_sf, *zsx, *zsf_t, *asf_t;
  float *w13_g, *w2_g;
  int sf_tiles;
  // the step before the tail (optional): [W_lat | W_gate | zero rows] bf16, tile-major,
  // proj_rows x H, and its outputs
  __nv_bfloat16 *w_proj, *zp;
  float* lgp;
  int proj_rows;
  int dep_routed, dep_ntiles;
  int cap, max_hist_blocks;
  bool wide_ok;  // token-major engine usable (dims and launch register count)
  // The combine buffer r must be all zero when a forward starts: each norm row zeroes its
  // row of r after reading it.  A forward that copies r out (debug) leaves it in place,
  // as may one that stopped early; the next forward then clears it whole first.
  bool r_dirty;
  // descriptors per BN variant (token-side maps depend on the box height)
  CUtensorMap tm_zqp[kNumBN], tm_aq[kNumBN], tm_n[kNumBN], tm_as[kNumBN];
  void* allocs[64];
  int nallocs;
};

namespace {

cudaError_t halloc(klt_handle* h, void** p, size_t bytes) {
  if (h->nallocs >= static_cast<int>(sizeof(h->allocs) / sizeof(h->allocs[0])))
    return cudaErrorMemoryAllocation;
  cudaError_t e = cudaMalloc(p, bytes < 256 ? 256 : bytes);
  if (e != cudaSuccess) return e;
  h->allocs[h->nallocs++] = *p;
  return cudaMemset(*p, 0, bytes < 256 ? 256 : bytes);
}

void free_all(klt_handle* h) {
  for (int i = 0; i < h->nallocs; ++i) cudaFree(h->allocs[i]);
  h->nallocs = 0;
}

int check_dims(const klt_dims* d) {
  if (!(d->eps > 0.f) || d->eps > 1.f || d->max_tokens < 1 || d->E < 1 || d->topk < 1)
    return KLT_ERR_INVALID_ARG;
  if (d->H <= 0 || d->L <= 0 || d->I <= 0 || d->Is <= 0) return KLT_ERR_INVALID_ARG;
  if (d->H % 128 || d->L % 128 || d->I % 128 || d->Is % 128) return KLT_ERR_UNSUPPORTED;
  if (d->E > MAX_E || d->topk > d->E || d->topk > MAX_TOPK) return KLT_ERR_UNSUPPORTED;
  if (d->L > 128 * MAX_KB || d->I > 128 * MAX_KB) return KLT_ERR_UNSUPPORTED;
  if (d->routed_fmt != KLT_FMT_FP8_B128 && d->routed_fmt != KLT_FMT_NVFP4 &&
      d->routed_fmt != KLT_FMT_MXFP8 && d->routed_fmt != KLT_FMT_NVFP4_W4A4)
    return KLT_ERR_UNSUPPORTED;
  // MXFP8 runs on the token-major engine only (256-wide units)
  if (d->routed_fmt == KLT_FMT_MXFP8 && (d->H % 256 || d->L % 256)) return KLT_ERR_UNSUPPORTED;
  // so does NVFP4_W4A4, whose k-blocks are 256 e2m1 values (L and I are GEMM K extents)
  if (d->routed_fmt == KLT_FMT_NVFP4_W4A4 && (d->H % 256 || d->L % 256 || d->I % 256))
    return KLT_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(d->max_tokens) * d->topk > (1 << 20)) return KLT_ERR_UNSUPPORTED;
  return KLT_OK;
}

// Routing of a small batch in one launch (route_small_kernel): the feature-major engine,
// one permutation block of at most SMALL_PAIRS pairs, e4m3 activations with fp32 scales.
bool small_routing(const klt_handle* h, int M, bool wide) {
  const bool bs = h->d.routed_fmt == KLT_FMT_MXFP8 || h->d.routed_fmt == KLT_FMT_NVFP4_W4A4;
  return !wide && !bs && static_cast<long long>(M) * h->d.topk <= SMALL_PAIRS;
}

// Token-tile width: the smallest tile that holds a decode batch, 64 beyond that (the
// 128-wide tile is kept for explicit selection).
int bn_index(int M, int force_bn) {
  for (int i = 0; i < kNumBN; ++i)
    if (force_bn == kBN[i]) return i;
  return M <= 16 ? 0 : (M <= 32 ? 1 : 2);
}

// k splits for a non-routed task so that a launch has enough units to fill the GPU,
// keeping split-K partial traffic small next to the weight bytes.
void plan_split(GemmTask& T, int ntiles, int target_units, int bn) {
  const int tiles = ntiles * T.ftiles;
  int ks = 1;
  if (tiles < target_units) {
    ks = (target_units + tiles - 1) / tiles;
    const int min_kb = std::max(4, bn / 8);
    ks = std::min(ks, std::max(1, T.kb_total / min_kb));
    while (ks > 1 && tiles * ks > kMaxSplitUnits) --ks;
  }
  T.kb_per_split = (T.kb_total + ks - 1) / ks;
  T.ksplit = (T.kb_total + T.kb_per_split - 1) / T.kb_per_split;
  T.ntiles = ntiles;
  T.units = ntiles * T.ftiles * T.ksplit;
}

}  // namespace

extern "C" {

const char* klt_strerror(int code) {
  switch (code) {
    case KLT_OK: return "ok";
    case KLT_ERR_INVALID_ARG: return "invalid argument";
    case KLT_ERR_UNSUPPORTED: return "unsupported shape, format or device";
    case KLT_ERR_ALIGN: return "pointer not 16-byte aligned";
    case KLT_ERR_CUDA: return "CUDA call failed";
    case KLT_ERR_DEVICE_TIMEOUT: return "bounded device wait expired";
    case KLT_ERR_OOM: return "device allocation failed";
    case KLT_ERR_TOO_LARGE: return "request exceeds the fixed scratch capacity";
    default: return "unknown status";
  }
}

int klt_create(const klt_dims* d, const klt_weights* w, uint32_t flags, klt_handle** out) {
  if (!out) return KLT_ERR_INVALID_ARG;
  *out = nullptr;
  if (!d || !w) return KLT_ERR_INVALID_ARG;
  int rc = check_dims(d);
  if (rc) return rc;
  if ((flags & KLT_FLAG_DETERMINISTIC) && (flags & KLT_FLAG_PHASED)) return KLT_ERR_UNSUPPORTED;
  const bool nvfp4 = d->routed_fmt == KLT_FMT_NVFP4;
  const bool mx = d->routed_fmt == KLT_FMT_MXFP8;
  const bool nv4 = d->routed_fmt == KLT_FMT_NVFP4_W4A4;  // packed FP4 x FP4, block-scaled
  if ((mx || nv4) && (flags & KLT_FLAG_PHASED)) return KLT_ERR_UNSUPPORTED;
  if ((nvfp4 || nv4) && (!w->w13_global || !w->w2_global)) return KLT_ERR_INVALID_ARG;
  if ((nvfp4 || nv4) && (!aligned16(w->w13_global) || !aligned16(w->w2_global)))
    return KLT_ERR_ALIGN;
  if ((w->w_lat == nullptr) != (w->w_gate == nullptr)) return KLT_ERR_INVALID_ARG;
  if (w->w_lat && (!aligned16(w->w_lat) || !aligned16(w->w_gate))) return KLT_ERR_ALIGN;
  const void* ptrs[] = {w->w13, w->w13_scale, w->w2, w->w2_scale, w->ws13, w->ws2,
                        w->w_up, w->gamma};
  for (const void* p : ptrs)
    if (!p) return KLT_ERR_INVALID_ARG;
  for (const void* p : ptrs)
    if (!aligned16(p)) return KLT_ERR_ALIGN;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KLT_ERR_CUDA;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return KLT_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return KLT_ERR_UNSUPPORTED;
  if (!get_encode()) return KLT_ERR_CUDA;
  if (!gemm_regs_ok()) return KLT_ERR_UNSUPPORTED;

  klt_handle* h = new (std::nothrow) klt_handle();
  if (!h) return KLT_ERR_OOM;
  std::memset(h, 0, sizeof(*h));
  h->d = *d;
  h->flags = flags;
  h->device = dev;
  h->num_sms = prop.multiProcessorCount;
  const int64_t E = d->E, H = d->H, L = d->L, I = d->I, Is = d->Is, k = d->topk;
  const int64_t Mx = d->max_tokens;
  h->cap = static_cast<int>(Mx * k);
  h->max_hist_blocks = (h->cap + PERM_BLOCK - 1) / PERM_BLOCK;
  const int64_t cap = h->cap;

#define KLT_ALLOC(ptr, bytes)                                                   \
  do {                                                                          \
    if (halloc(h, reinterpret_cast<void**>(&(ptr)), (bytes)) != cudaSuccess) {  \
      free_all(h);                                                              \
      delete h;                                                                 \
      return KLT_ERR_OOM;                                                       \
    }                                                                           \
  } while (0)
  // NVFP4 weights are held as their exact bf16 values (2 bytes per weight), except in the
  // FP4 x FP4 format, which keeps them packed (two per byte)
  const int64_t w13_bytes = nvfp4 ? E * 2 * I * L * 2 : (nv4 ? E * 2 * I * L / 2 : E * 2 * I * L);
  const int64_t w2_bytes = nvfp4 ? E * L * I * 2 : (nv4 ? E * L * I / 2 : E * L * I);
  KLT_ALLOC(h->w13, w13_bytes);
  KLT_ALLOC(h->w13_s, E * (2 * I / 128) * (L / 128) * 4);
  KLT_ALLOC(h->w2, w2_bytes);
  KLT_ALLOC(h->w2_s, E * (L / 128) * (I / 128) * 4);
  KLT_ALLOC(h->ws13, 2 * Is * H * 2);
  KLT_ALLOC(h->ws2, H * Is * 2);
  KLT_ALLOC(h->w_up, H * L * 2);
  KLT_ALLOC(h->gamma, L * 2);
  KLT_ALLOC(h->ids, cap * 4);
  KLT_ALLOC(h->wts, cap * 4);
  KLT_ALLOC(h->wperm, cap * 4);
  KLT_ALLOC(h->pos, cap * 4);
  KLT_ALLOC(h->gidx, cap * 4);
  KLT_ALLOC(h->slot, cap * 4);
  KLT_ALLOC(h->hist, static_cast<int64_t>(h->max_hist_blocks) * E * 4);
  KLT_ALLOC(h->cnt, E * 4);
  KLT_ALLOC(h->off, (E + 1) * 4);
  KLT_ALLOC(h->tile_off, (E + 1) * 4);
  KLT_ALLOC(h->zq, Mx * L);
  KLT_ALLOC(h->zs, Mx * (L / 128) * 4);
  KLT_ALLOC(h->zq_perm, nvfp4 ? 16 : cap * L);
  if (nvfp4) {
    KLT_ALLOC(h->zqb_perm, cap * L * 2);
    KLT_ALLOC(h->aqb, cap * I * 2);
  }
  KLT_ALLOC(h->zsT, (L / 128) * cap * 4);
  KLT_ALLOC(h->aq, cap * I);
  KLT_ALLOC(h->asT, (I / 128) * cap * 4);
  KLT_ALLOC(h->r, Mx * L * 4);
  if (flags & KLT_FLAG_DETERMINISTIC) KLT_ALLOC(h->yw, cap * L * 4);
  KLT_ALLOC(h->n, Mx * L * 2);
  KLT_ALLOC(h->a_s, Mx * Is * 2);
  // split-K partials: [shared L1 | output GEMM], one half each
  KLT_ALLOC(h->ws, 2LL * kMaxSplitUnits * 2 * 128 * 128 * 4);
  KLT_ALLOC(h->split_cnt, 2LL * kMaxCounters * 4);
  KLT_ALLOC(h->out_acc, static_cast<int64_t>(kWideSplitMaxTiles) * 128 * H * 4);
  KLT_ALLOC(h->out_cnt, static_cast<int64_t>(kWideSplitMaxTiles) * (H / 128) * 4);
  KLT_ALLOC(h->sched, 64 * 4);
  h->dep_routed = static_cast<int>((cap + 15) / 16 + E);
  h->dep_ntiles = static_cast<int>((Mx + 15) / 16);
  KLT_ALLOC(h->dep_cnt, (static_cast<int64_t>(h->dep_routed) + 1 + 2 * h->dep_ntiles) * 4);
  KLT_ALLOC(h->err, 256);
  if (mx || nv4) {
    // one scale byte per sf_group K-elements of a row; 512-byte tiles of 4 bytes x 128 rows
    const int64_t g = mx ? 32 : 16;
    h->sf_tiles = static_cast<int>(cap / 128 + E);
    KLT_ALLOC(h->w13_sf, E * 2 * I * (L / g));
    KLT_ALLOC(h->w2_sf, E * L * (I / g));
    KLT_ALLOC(h->zsx, Mx * (L / g));
    KLT_ALLOC(h->zsf_t, static_cast<int64_t>(h->sf_tiles) * (L / (4 * g)) * 512);
    KLT_ALLOC(h->asf_t, static_cast<int64_t>(h->sf_tiles) * (I / (4 * g)) * 512);
  }
  if (nv4) {  // the weights' fp32 per-matrix scales, applied in the epilogue
    KLT_ALLOC(h->w13_g, E * 4);
    KLT_ALLOC(h->w2_g, E * 4);
  }
  if (w->w_lat) {
    // rows: W_lat (L), W_gate (E), zero rows up to a multiple of 128 (one output tile)
    h->proj_rows = static_cast<int>((L + E + 127) / 128 * 128);
    KLT_ALLOC(h->w_proj, static_cast<int64_t>(h->proj_rows) * H * 2);
    KLT_ALLOC(h->zp, Mx * L * 2);
    KLT_ALLOC(h->lgp, Mx * E * 4);
  }
#undef KLT_ALLOC

  // Weights are copied tile-major (one contiguous 16 KB block per 128 rows x 128 bytes of
  // K), so every TMA box of a weight operand is a single contiguous DRAM stream.
  bool ok = true;
  if (nvfp4) {
    // exact bf16 values e2m1 * e4m3 block scale; the fp32 matrix scale becomes the
    // promotion scale of every 128-wide K group
    ok &= launch_nvfp4_expand(static_cast<const uint8_t*>(w->w13),
                              static_cast<const uint8_t*>(w->w13_scale), h->w13, E * 2 * I, L,
                              0) == cudaSuccess;
    ok &= launch_nvfp4_expand(static_cast<const uint8_t*>(w->w2),
                              static_cast<const uint8_t*>(w->w2_scale), h->w2, E * L, I,
                              0) == cudaSuccess;
    ok &= launch_fill_expert_scale(w->w13_global, h->w13_s, static_cast<int>(E),
                                   (2 * I / 128) * (L / 128), 0) == cudaSuccess;
    ok &= launch_fill_expert_scale(w->w2_global, h->w2_s, static_cast<int>(E),
                                   (L / 128) * (I / 128), 0) == cudaSuccess;
  } else {  // e4m3 codes, or packed e2m1 (the same 128-byte k-blocks of a row)
    ok &= launch_tile_relayout(w->w13, h->w13, E * 2 * I, nv4 ? L / 2 : L, 0) == cudaSuccess;
    ok &= launch_tile_relayout(w->w2, h->w2, E * L, nv4 ? I / 2 : I, 0) == cudaSuccess;
  }
  if (mx || nv4) {
    const int64_t g = mx ? 32 : 16;
    ok &= launch_sf_relayout(static_cast<const uint8_t*>(w->w13_scale), h->w13_sf, E * 2 * I,
                             L / g, 0) == cudaSuccess;
    ok &= launch_sf_relayout(static_cast<const uint8_t*>(w->w2_scale), h->w2_sf, E * L, I / g,
                             0) == cudaSuccess;
  }
  if (nv4) {
    ok &= cudaMemcpy(h->w13_g, w->w13_global, E * 4, cudaMemcpyDeviceToDevice) == cudaSuccess;
    ok &= cudaMemcpy(h->w2_g, w->w2_global, E * 4, cudaMemcpyDeviceToDevice) == cudaSuccess;
  }
  ok &= launch_tile_relayout(w->ws13, h->ws13, 2 * Is, H * 2, 0) == cudaSuccess;
  ok &= launch_tile_relayout(w->ws2, h->ws2, H, Is * 2, 0) == cudaSuccess;
  ok &= launch_tile_relayout(w->w_up, h->w_up, H, L * 2, 0) == cudaSuccess;
  if (w->w_lat) {
    ok &= launch_tile_relayout(w->w_lat, h->w_proj, L, H * 2, 0) == cudaSuccess;
    // the gate rows and the zero rows after them, as one block of 128-row tiles
    const int64_t gate_rows = h->proj_rows - L;
    void* tmp = nullptr;
    if (cudaMalloc(&tmp, gate_rows * H * 2) != cudaSuccess) {
      free_all(h);
      delete h;
      return KLT_ERR_OOM;
    }
    ok &= cudaMemset(tmp, 0, gate_rows * H * 2) == cudaSuccess;
    ok &= cudaMemcpy(tmp, w->w_gate, E * H * 2, cudaMemcpyDeviceToDevice) == cudaSuccess;
    ok &= launch_tile_relayout(tmp, reinterpret_cast<uint8_t*>(h->w_proj) + L * H * 2,
                               gate_rows, H * 2, 0) == cudaSuccess;
    ok &= cudaDeviceSynchronize() == cudaSuccess;
    cudaFree(tmp);
  }
  if (!nvfp4 && !mx && !nv4) {
    ok &= cudaMemcpy(h->w13_s, w->w13_scale, E * (2 * I / 128) * (L / 128) * 4,
                     cudaMemcpyDeviceToDevice) == cudaSuccess;
    ok &= cudaMemcpy(h->w2_s, w->w2_scale, E * (L / 128) * (I / 128) * 4,
                     cudaMemcpyDeviceToDevice) == cudaSuccess;
  }
  ok &= cudaMemcpy(h->gamma, w->gamma, L * 2, cudaMemcpyDeviceToDevice) == cudaSuccess;

  const CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUtensorMapDataType BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  for (int b = 0; b < kNumBN; ++b) {
    if (nvfp4) {
      ok &= encode_2d(&h->tm_zqp[b], h->zqb_perm, BF, 2, cap, L, kBN[b]);
      ok &= encode_2d(&h->tm_aq[b], h->aqb, BF, 2, cap, I, kBN[b]);
    } else {  // byte rows: e4m3 codes, or e2m1 codes two per byte
      ok &= encode_2d(&h->tm_zqp[b], h->zq_perm, U8, 1, cap, nv4 ? L / 2 : L, kBN[b]);
      ok &= encode_2d(&h->tm_aq[b], h->aq, U8, 1, cap, nv4 ? I / 2 : I, kBN[b]);
    }
    ok &= encode_2d(&h->tm_n[b], h->n, BF, 2, Mx, L, kBN[b]);
    ok &= encode_2d(&h->tm_as[b], h->a_s, BF, 2, Mx, Is, kBN[b]);
  }
  if (!ok || cudaDeviceSynchronize() != cudaSuccess) {
    free_all(h);
    delete h;
    return KLT_ERR_CUDA;
  }
  h->wide_ok = L % 256 == 0 && H % 256 == 0 && wide_regs_ok(wide_kernel_regs());
  if ((mx || nv4) && !h->wide_ok) {
    free_all(h);
    delete h;
    return KLT_ERR_UNSUPPORTED;
  }
  *out = h;
  return KLT_OK;
}

int klt_launch_count(const klt_handle* h, int32_t M) {
  if (!h || M <= 0) return 0;
  const int nblocks = (M * h->d.topk + PERM_BLOCK - 1) / PERM_BLOCK;
  // phased: 3 GEMMs + norm; block-scaled layers: routed and dense launches
  const bool bs = h->d.routed_fmt == KLT_FMT_MXFP8 || h->d.routed_fmt == KLT_FMT_NVFP4_W4A4;
  const int gemm_launches = (h->flags & KLT_FLAG_PHASED) ? 4 : (bs ? 2 : 1);
  const int routing = small_routing(h, M, klt_gemm_tile(h, M, 0) == 256)
                          ? 1
                          : 3 + (nblocks > 1 ? 1 : 0);
  return routing + gemm_launches;
}

int klt_gemm_tile(const klt_handle* h, int32_t M, int32_t force_bn) {
  if (!h) return -KLT_ERR_INVALID_ARG;
  const bool phased = (h->flags & KLT_FLAG_PHASED) != 0;
  // block-scaled units exist in the token-major engine only
  if (h->d.routed_fmt == KLT_FMT_MXFP8 || h->d.routed_fmt == KLT_FMT_NVFP4_W4A4)
    return (force_bn == 0 || force_bn == 256) && h->wide_ok && !phased ? 256
                                                                      : -KLT_ERR_UNSUPPORTED;
  if (force_bn == 256) return h->wide_ok && !phased ? 256 : -KLT_ERR_UNSUPPORTED;
  if (force_bn == 0 && h->wide_ok && !phased && M >= kWideMinTokens) return 256;
  return kBN[bn_index(M, force_bn)];
}

}  // extern "C"

namespace {

// One forward: the tail on (x, z, logits), or, with `from_hidden`, the projection of x into
// the handle's z and logits first.
int forward_impl(klt_handle* h, const void* x, const void* z, const float* logits, int32_t M,
                 void* out, klt_routing* ro, klt_debug* dbg, void* stream, bool from_hidden) {
  if (!h) return KLT_ERR_INVALID_ARG;
  if (M < 0 || M > h->d.max_tokens) return KLT_ERR_INVALID_ARG;
  if (from_hidden && !h->w_proj) return KLT_ERR_UNSUPPORTED;
  if (M == 0) return KLT_OK;
  if (from_hidden) {
    z = h->zp;
    logits = h->lgp;
  }
  if (!x || !z || !logits || !out) return KLT_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(z) || !aligned16(logits) || !aligned16(out))
    return KLT_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool pdl = !(h->flags & KLT_FLAG_NO_PDL);
  const klt_dims& d = h->d;
  const int E = d.E, k = d.topk, L = d.L, I = d.I, Is = d.Is, H = d.H;
  const bool phased = (h->flags & KLT_FLAG_PHASED) != 0;
  const int tile = klt_gemm_tile(h, M, dbg ? dbg->force_bn : 0);
  if (tile < 0) return -tile;
  const bool wide = tile == 256;
  const int bi = wide ? kNumBN - 1 : bn_index(M, tile);
  const int BN = kBN[bi];
  const bool nvfp4 = d.routed_fmt == KLT_FMT_NVFP4;
  const bool mx = d.routed_fmt == KLT_FMT_MXFP8;
  const bool nv4 = d.routed_fmt == KLT_FMT_NVFP4_W4A4;
  // routed K elements per 128-byte k-block: bf16 images, e4m3 codes, or e2m1 pairs
  const int rkb = nvfp4 ? 64 : (nv4 ? 256 : 128);
  const int Mk = M * k;
  const int nblocks = (Mk + PERM_BLOCK - 1) / PERM_BLOCK;
  const long long timeout_cycles =
      static_cast<long long>(dbg && dbg->timeout_ms > 0 ? dbg->timeout_ms : 1000) * 2000000LL;
  int launch = 0;
  auto mark = [&]() {
    if (dbg && launch < 8 && dbg->events[launch])
      cudaEventRecord(static_cast<cudaEvent_t>(dbg->events[launch]), s);
    ++launch;
  };
#define KLT_LAUNCH(expr)                      \
  do {                                        \
    if ((expr) != cudaSuccess) return KLT_ERR_CUDA; \
    mark();                                   \
  } while (0)

  // ---- the step before the tail: [z | logits] = x . [W_lat | W_gate]^T (feature-major
  // engine, split in K to fill the GPU; its tile counter was zeroed by the previous
  // forward's routing kernel or at create)
  if (from_hidden) {
    const int pbn = kBN[bn_index(M, 0)];
    GemmParams gpj;
    std::memset(&gpj, 0, sizeof(gpj));
    gpj.ntasks = 1;
    gpj.M = M;
    gpj.E = E;
    gpj.L = L;
    gpj.I = I;
    gpj.Is = Is;
    gpj.H = H;
    gpj.cap = h->cap;
    gpj.tile_off = h->tile_off;
    gpj.off = h->off;
    gpj.ws = h->ws;
    gpj.cnt = h->split_cnt;
    gpj.sched = h->sched + 6;
    gpj.err = h->err;
    gpj.timeout = timeout_cycles;
    gpj.zp = h->zp;
    gpj.lgp = h->lgp;
    GemmTask& P = gpj.task[0];
    P.kind = TASK_PROJ;
    P.a_rb_step = 1;
    P.ftiles = h->proj_rows / 128;
    P.kb_total = H / 64;
    P.kb_split0 = P.kb_total;
    P.a_kb[0] = P.a_kb[1] = H / 64;
    P.a_ptr[0] = P.a_ptr[1] = reinterpret_cast<const uint8_t*>(h->w_proj);
    if (!encode_2d(&P.tmB[0], x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, M, H, pbn))
      return KLT_ERR_CUDA;
    P.tmB[1] = P.tmB[0];
    // split in K so that the units fill the SMs in one wave (a second wave doubles the
    // launch's time at decode sizes); single 128-row tiles keep the partials that the last
    // arriver of a tile sums small (a split of 5 at decode: 5 x 8 KB per tile)
    {
      const int pt = (M + pbn - 1) / pbn;
      const int tiles = pt * P.ftiles;
      int ks = std::max(1, std::min(P.kb_total / 4, h->num_sms / std::max(1, tiles)));
      while (ks > 1 && tiles * ks > kMaxSplitUnits) --ks;
      P.kb_per_split = (P.kb_total + ks - 1) / ks;
      P.ksplit = (P.kb_total + P.kb_per_split - 1) / P.kb_per_split;
      P.ntiles = pt;
      P.units = tiles * P.ksplit;
    }
    KLT_LAUNCH(launch_gemm(gpj, pbn, h->num_sms, s, pdl));
  }

  // ---- K0: routing + latent quantisation + zero r + zero tile counters
  RouteParams rp;
  rp.logits = logits;
  rp.z = static_cast<const __nv_bfloat16*>(z);
  rp.ids = h->ids;
  rp.wts = h->wts;
  rp.zq = h->zq;
  rp.zs = h->zs;
  rp.r = h->r;
  rp.sched = h->sched;
  rp.nsched = 8;
  rp.zero_buf = h->dep_cnt;
  rp.zero_n = (h->flags & KLT_FLAG_PHASED) ? 0 : h->dep_routed + 1 + 2 * h->dep_ntiles;
  rp.M = M;
  rp.E = E;
  rp.k = k;
  rp.L = L;
  rp.bs = mx ? BS_MX8 : (nv4 ? BS_NV4 : BS_NONE);
  rp.zsx = h->zsx;
  // r is zeroed by the norm rows unless the caller copies the combine buffer out afterwards
  const bool keep_r = dbg && dbg->r && !(h->flags & KLT_FLAG_DETERMINISTIC);
  if (h->r_dirty) {
    if (cudaMemsetAsync(h->r, 0, static_cast<size_t>(d.max_tokens) * L * 4, s) != cudaSuccess)
      return KLT_ERR_CUDA;
    h->r_dirty = false;
  }
  const bool r_left = keep_r;  // after this forward r holds the combine, or zeros
  h->r_dirty = true;           // until every launch of this forward is issued

  // ---- K1: permutation
  PermParams pp;
  pp.ids = h->ids;
  pp.hist = h->hist;
  pp.cnt = h->cnt;
  pp.off = h->off;
  pp.tile_off = h->tile_off;
  pp.gidx = h->gidx;
  pp.slot = h->slot;
  pp.pos = h->pos;
  pp.zq = h->zq;
  pp.zs = h->zs;
  pp.zq_perm = h->zq_perm;
  pp.zqb_perm = nvfp4 ? h->zqb_perm : nullptr;
  pp.zsT = h->zsT;
  pp.wts = h->wts;
  pp.wperm = h->wperm;
  pp.M = M;
  pp.E = E;
  pp.k = k;
  pp.L = L;
  pp.cap = h->cap;
  pp.bn = BN;  // routed tile list in BN-token tiles (128 for the token-major engine)
  pp.nblocks = nblocks;
  pp.zsx = h->zsx;
  pp.zsf_t = (mx || nv4) ? h->zsf_t : nullptr;
  pp.sf_tiles = h->sf_tiles;
  pp.sf_group = mx ? 32 : 16;
  pp.zrow = nv4 ? L / 2 : L;
  if (small_routing(h, M, wide)) {
    KLT_LAUNCH(launch_route_small(rp, pp, s, pdl));
  } else {
    KLT_LAUNCH(launch_route(rp, s, pdl));
    if (nblocks > 1) KLT_LAUNCH(launch_perm_hist(pp, s, pdl));
    KLT_LAUNCH(launch_perm_scatter(pp, s, pdl));
    KLT_LAUNCH(launch_perm_gather(pp, s, pdl));
  }

  // ---- common GEMM parameters
  GemmParams gp;
  std::memset(&gp, 0, sizeof(gp));
  gp.M = M;
  gp.E = E;
  gp.L = L;
  gp.I = I;
  gp.Is = Is;
  gp.H = H;
  gp.cap = h->cap;
  gp.tile_off = h->tile_off;
  gp.off = h->off;
  gp.gidx = h->gidx;
  gp.wperm = h->wperm;
  gp.zsT = h->zsT;
  gp.w13_s = h->w13_s;
  gp.w2_s = h->w2_s;
  gp.aq = h->aq;
  gp.aqb = nvfp4 ? h->aqb : nullptr;
  gp.asT = h->asT;
  gp.r = h->r;
  gp.zero_r = keep_r ? 0 : 1;
  gp.yw = (h->flags & KLT_FLAG_DETERMINISTIC) ? h->yw : nullptr;
  gp.pos = h->pos;
  gp.topk = k;
  gp.a_s = h->a_s;
  gp.out = static_cast<__nv_bfloat16*>(out);
  gp.ws = h->ws;
  gp.cnt = h->split_cnt;
  gp.err = h->err;
  gp.timeout = timeout_cycles;
  gp.trace_n = dbg ? dbg->trace_entries : 0;
  long long* trace = (dbg && dbg->trace && dbg->trace_entries > 0)
                         ? reinterpret_cast<long long*>(dbg->trace) : nullptr;
  const long long trace_launch = static_cast<long long>(h->num_sms) * 4 * gp.trace_n;
  const int ntiles = (M + BN - 1) / BN;
  const int grid = h->num_sms;
  const size_t ws_task = static_cast<size_t>(kMaxSplitUnits) * 2 * 128 * 128;

  const bool fused = !phased;
  if (wide) {
    // Token-major engine: 128-token tiles, 256 features per unit, the five tasks of the
    // fused launch with the same dependency counters.
    GemmParams gw = gp;
    gw.ntasks = 5;
    // prefill-size batches: pairs of token tiles share each staged weight tile of the
    // BF16 tasks (3 stages of 64 KB); otherwise 4 stages of 48 KB
    const bool dual = ntiles >= kDualMinTiles;
    gw.asf_t = h->asf_t;
    gw.w_stages = dual ? 3 : 4;
    gw.w_stage_bytes = dual ? 64 * 1024 : 48 * 1024;
    gw.sched = h->sched + 3;
    gw.stall_after = dbg ? dbg->stall_after_kblocks : 0;
    gw.trace = trace;
    GemmTask& R = gw.task[0];  // routed L1: gate and up row blocks of one 128-output tile
    R.kind = TASK_ROUTED_L1;
    R.fp8 = !nvfp4;  // byte operands (e4m3, or e2m1 pairs)
    R.kpg = (mx || nv4) ? 0 : (nvfp4 ? 2 : 1);  // block-scaled: the tensor core scales
    R.routed = 1;
    R.ftiles = I / 128;
    R.kb_total = L / rkb;
    R.kb_split0 = R.kb_total;
    R.ksplit = 1;
    R.kb_per_split = R.kb_total;
    R.a_rb_up = I / 128;
    R.a_rb_expert = 2 * I / 128;
    R.a_kb[0] = R.a_kb[1] = L / rkb;
    R.a_ptr[0] = R.a_ptr[1] = h->w13;
    R.tmB[0] = R.tmB[1] = h->tm_zqp[bi];
    R.a_sf = (mx || nv4) ? h->w13_sf : nullptr;
    R.t_sf = (mx || nv4) ? h->zsf_t : nullptr;
    R.a_g = nv4 ? h->w13_g : nullptr;
    GemmTask& S = gw.task[1];  // shared L1 (bf16)
    S.kind = TASK_SHARED_L1;
    S.ftiles = Is / 128;
    S.kb_total = H / 64;
    S.kb_split0 = S.kb_total;
    S.ksplit = 1;
    S.kb_per_split = S.kb_total;
    S.a_rb_up = Is / 128;
    S.a_kb[0] = S.a_kb[1] = H / 64;
    S.a_ptr[0] = S.a_ptr[1] = reinterpret_cast<const uint8_t*>(h->ws13);
    S.ntiles = ntiles;
    S.dual = dual;
    S.units = (S.dual ? (ntiles + 1) / 2 : ntiles) * S.ftiles;
    if (!encode_2d(&S.tmB[0], x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, M, H, BN))
      return KLT_ERR_CUDA;
    S.tmB[1] = S.tmB[0];
    GemmTask& R2 = gw.task[2];  // routed L2 + combine: two row blocks of W2 per unit
    R2.kind = TASK_ROUTED_L2;
    R2.fp8 = !nvfp4;
    R2.kpg = (mx || nv4) ? 0 : (nvfp4 ? 2 : 1);
    R2.a_sf = (mx || nv4) ? h->w2_sf : nullptr;
    R2.t_sf = (mx || nv4) ? h->asf_t : nullptr;
    R2.a_g = nv4 ? h->w2_g : nullptr;
    R2.routed = 1;
    R2.ftiles = L / 256;
    R2.kb_total = I / rkb;
    R2.kb_split0 = R2.kb_total;
    R2.ksplit = 1;
    R2.kb_per_split = R2.kb_total;
    R2.a_rb_expert = L / 128;
    R2.a_kb[0] = R2.a_kb[1] = I / rkb;
    R2.a_ptr[0] = R2.a_ptr[1] = h->w2;
    R2.tmB[0] = R2.tmB[1] = h->tm_aq[bi];
    R2.dep = DEP_L1_TILE;
    GemmTask& N = gw.task[3];  // RMSNorm, one token row per unit
    N.kind = TASK_NORM;
    N.dep = DEP_ALL_L2;
    N.ftiles = 1;
    N.ksplit = 1;
    N.ntiles = ntiles;
    N.units = (M + kWideNormRows - 1) / kWideNormRows;  // a token row per epilogue warp
    N.tmB[0] = N.tmB[1] = h->tm_n[bi];
    GemmTask& O = gw.task[4];  // out = bf16([n | a_s] . [W_up | Ws2]^T), 256 outputs per unit
    O.kind = TASK_OUT;
    O.ftiles = H / 256;
    O.kb_total = L / 64 + Is / 64;
    O.kb_split0 = L / 64;
    O.a_kb[0] = L / 64;
    O.a_kb[1] = Is / 64;
    O.ksplit = 1;
    O.kb_per_split = O.kb_total;
    O.ntiles = ntiles;
    O.dual = dual;
    O.units = (O.dual ? (ntiles + 1) / 2 : ntiles) * O.ftiles;
    O.dep = DEP_OUT_TILE;
    // A batch of one or two token tiles has few output units, and they run after the norm
    // on few SMs: split them in K (at least 8 k-blocks each) so that one wave of units
    // covers the GPU.  The splits add into out_acc and the last of a tile rounds it (not
    // with the fixed-order combine, whose output stays bitwise reproducible).
    if (!dual && ntiles <= kWideSplitMaxTiles && !(h->flags & KLT_FLAG_DETERMINISTIC)) {
      const int tiles = ntiles * O.ftiles;
      const int ks = std::min(grid / tiles, O.kb_total / 8);
      if (ks > 1) {
        O.kb_per_split = (O.kb_total + ks - 1) / ks;
        O.ksplit = (O.kb_total + O.kb_per_split - 1) / O.kb_per_split;
        O.units = tiles * O.ksplit;
      }
    }
    gw.out_acc = h->out_acc;
    gw.out_cnt = h->out_cnt;
    O.a_ptr[0] = reinterpret_cast<const uint8_t*>(h->w_up);
    O.a_ptr[1] = reinterpret_cast<const uint8_t*>(h->ws2);
    O.tmB[0] = h->tm_n[bi];
    O.tmB[1] = h->tm_as[bi];
    std::swap(gw.task[0], gw.task[1]);  // shared L1 first (its weights are prefetched)
    gw.pf_ptr = reinterpret_cast<const uint8_t*>(h->ws13);
    gw.pf_bytes = 2LL * Is * H * 2;
    gw.l1_done = h->dep_cnt;
    gw.l2_done = h->dep_cnt + h->dep_routed;
    gw.norm_done = gw.l2_done + 1;
    gw.sh_done = gw.norm_done + h->dep_ntiles;
    gw.l1_target = I / 128;
    gw.sh_target = Is / 128;
    gw.l2_ftiles = L / 256;
    gw.gamma = h->gamma;
    gw.nrm = h->n;
    gw.eps = d.eps;
    if (!mx && !nv4) {
      KLT_LAUNCH(launch_wide(gw, grid, s, pdl));
    } else {
      // Block-scaled layers: the routed units keep one accumulator slot (their scale ring
      // takes the other half of TMEM), so they run as a launch of their own; the BF16
      // shared L1, norm and output GEMM follow in a second launch with two slots and dual
      // token tiles.  The dependency counters carry over (zeroed once by routing).
      GemmParams gr = gw, gd = gw;
      gr.bs = mx ? BS_MX8 : BS_NV4;
      gr.ntasks = 2;
      gr.task[0] = gw.task[1];  // routed L1
      gr.task[1] = gw.task[2];  // routed L2
      // NVFP4: 3 stages that carry their 6 KB of scale tiles; MX: 4 of 48 KB
      gr.w_stages = nv4 ? 3 : 4;
      gr.w_stage_bytes = nv4 ? 48 * 1024 + 6 * 1024 : 48 * 1024;
      gr.pf_ptr = nullptr;
      gr.pf_bytes = 0;
      gd.bs = BS_NONE;
      gd.ntasks = 3;
      gd.task[0] = gw.task[0];  // shared L1
      gd.task[1] = gw.task[3];  // norm
      gd.task[2] = gw.task[4];  // output
      gd.sched = h->sched + 4;
      gd.pf_ptr = nullptr;
      gd.pf_bytes = 0;
      gd.trace = trace ? trace + trace_launch : nullptr;
      KLT_LAUNCH(launch_wide(gr, grid, s, pdl));
      KLT_LAUNCH(launch_wide(gd, grid, s, pdl));
    }
  } else {
    GemmParams g1 = gp, g2 = gp, g3 = gp;
    // ---- GEMM 1: shared L1 (bf16, split-K) + routed L1 (fp8, SwiGLU + act quant)
    {
      // Routed units first, then the shared expert in small k-splits that fill the tail.
      GemmTask& R = g1.task[0];
      R.kind = TASK_ROUTED_L1;
      R.fp8 = !nvfp4;
      R.kpg = nvfp4 ? 2 : 1;
      R.routed = 1;
      R.ftiles = I / 128;
      R.kb_total = L / rkb;
      R.kb_split0 = R.kb_total;
      // routed units stay whole in K (measured: a k-split's reduce costs more than the
      // balance it buys)
      R.ksplit = 1;
      R.kb_per_split = R.kb_total;
      R.pair = 1;
      R.a_rb_up = I / 128;
      R.a_rb_step = 1;
      R.a_rb_expert = 2 * I / 128;
      R.a_kb[0] = R.a_kb[1] = L / rkb;
      R.a_ptr[0] = R.a_ptr[1] = h->w13;
      R.tmB[0] = h->tm_zqp[bi];
      R.tmB[1] = h->tm_zqp[bi];
      GemmTask& S = g1.task[1];
      S.kind = TASK_SHARED_L1;
      S.routed = 0;
      S.ftiles = Is / 128;
      S.kb_total = H / 64;
      S.kb_split0 = S.kb_total;
      S.pair = 1;
      S.a_rb_up = Is / 128;
      S.a_rb_step = 1;
      S.a_kb[0] = S.a_kb[1] = H / 64;
      S.ws_tile_base = 0;
      S.ws_off = 0;
      // k splits of about 16 k-blocks: each split's partial and the last arrival's
      // fixed-order reduce cost more than the balance finer splits buy (measured: 8-block
      // splits 82 us at M=4 and 163 us at M=16, 16-block splits 75 and 162 us)
      plan_split(S, ntiles, ntiles * S.ftiles * std::max(1, S.kb_total / 16), BN);
      if (!encode_2d(&S.tmB[0], x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, M, H, BN))
        return KLT_ERR_CUDA;
      // A batch that touches few experts has fewer routed L1 units than SMs: split them in
      // K (whole promotion groups) so the routed weights stream through every SM.  The
      // splits' partials go to the workspace after the shared expert's; the last split of
      // a tile sums them in a fixed order and runs the SwiGLU/requantisation epilogue.
      {
        const int ntr_est = std::min(E, Mk);                   // touched experts, at most
        const int ntr_ub = ntr_est + (Mk + BN - 1) / BN;        // routed tiles, at most
        const int r_units = ntr_est * R.ftiles;
        const size_t tile_floats = 2ull * BN * 128;
        const size_t s_slots = static_cast<size_t>(S.units);
        const int base = S.ntiles * S.ftiles;
        int ks = r_units < grid ? (grid + r_units - 1) / r_units : 1;
        ks = std::min(ks, std::max(1, R.kb_total / (4 * R.kpg)));
        while (ks > 1 &&
               (s_slots + static_cast<size_t>(ntr_ub) * R.ftiles * ks) * tile_floats > ws_task)
          --ks;
        if (ks > 1 && base + ntr_ub * R.ftiles <= kMaxCounters) {
          const int groups = R.kb_total / R.kpg;
          R.kb_per_split = ((groups + ks - 1) / ks) * R.kpg;
          R.ksplit = (R.kb_total + R.kb_per_split - 1) / R.kb_per_split;
          R.ws_tile_base = base;
          R.ws_off = static_cast<long long>(s_slots * tile_floats);
        }
      }
      S.a_ptr[0] = S.a_ptr[1] = reinterpret_cast<const uint8_t*>(h->ws13);
      S.tmB[1] = S.tmB[0];
    }
    // ---- GEMM 2: routed L2 with the top-k weighted scatter-combine into r
    {
      GemmTask& R = g2.task[0];
      R.kind = TASK_ROUTED_L2;
      R.fp8 = !nvfp4;
      R.kpg = nvfp4 ? 2 : 1;
      R.routed = 1;
      // two consecutive 128-row blocks of W2 per unit (one 2 x BN accumulator slot per
      // k-block): half the MMA-issue bookkeeping per weight byte of single-tile units
      const bool r2pair = (L / 128) % 2 == 0;
      R.pair = r2pair ? 1 : 0;
      R.a_rb_up = 1;
      R.a_rb_step = r2pair ? 2 : 1;
      R.ftiles = r2pair ? L / 256 : L / 128;
      R.kb_total = I / rkb;
      R.kb_split0 = R.kb_total;
      R.ksplit = 1;
      R.kb_per_split = R.kb_total;
      R.a_rb_expert = L / 128;
      R.a_kb[0] = R.a_kb[1] = I / rkb;
      R.a_ptr[0] = R.a_ptr[1] = h->w2;
      R.tmB[0] = h->tm_aq[bi];
      R.tmB[1] = h->tm_aq[bi];
    }
    // ---- GEMM 3: out = bf16([n | a_s] . [W_up | Ws2]^T)
    {
      GemmTask& O = g3.task[0];
      O.kind = TASK_OUT;
      O.routed = 0;
      O.ftiles = H / 128;
      O.kb_total = L / 64 + Is / 64;
      O.kb_split0 = L / 64;
      O.ws_tile_base = 0;
      O.a_kb[0] = L / 64;
      O.a_kb[1] = Is / 64;
      O.ksplit = 1;
      O.kb_per_split = O.kb_total;
      O.ntiles = ntiles;
      O.units = ntiles * O.ftiles;
      if (fused) {
        // units come from the launch-wide counter, after the other tasks' units
        O.ws_tile_base = kMaxCounters;
        O.ws_off = static_cast<long long>(ws_task);
        plan_split(O, ntiles, 2 * grid, BN);
      } else if (O.units < 4 * grid) {
        // static stream-K: every CTA streams the same number of k-blocks (no more CTAs than
        // k-blocks, so every CTA's range is non-empty)
        O.streamk = 1;
        O.sk_total = static_cast<long long>(O.units) * O.kb_total;
        O.sk_grid = static_cast<int>(std::min<long long>(grid, O.sk_total));
      }
      O.a_ptr[0] = reinterpret_cast<const uint8_t*>(h->w_up);
      O.a_ptr[1] = reinterpret_cast<const uint8_t*>(h->ws2);
      O.tmB[0] = h->tm_n[bi];
      O.tmB[1] = h->tm_as[bi];
    }
    if (fused) {
      // One persistent launch: routed L1 and shared L1, routed L2 (after its token tile's L1
      // units), the RMSNorm (after every L2 unit) and the output GEMM (after its tile's norm
      // and shared L1), ordered so that every unit depends only on earlier units.
      GemmParams gf = gp;
      gf.ntasks = 5;
      gf.sched = h->sched + 3;
      gf.stall_after = dbg ? dbg->stall_after_kblocks : 0;
      gf.trace = trace;
      gf.cnt = h->split_cnt;
      // the shared L1 first: its weights were prefetched into L2 while routing ran, and its
      // tiles are done early for the output units over Ws2 (measured at 16 tokens: 172.5 ->
      // 165.6 us per step with the routed L1 first -> shared L1 first)
      gf.task[0] = g1.task[1];
      gf.task[1] = g1.task[0];
      gf.task[2] = g2.task[0];
      gf.task[2].dep = DEP_L1_TILE;
      GemmTask& N = gf.task[3];
      N.kind = TASK_NORM;
      N.dep = DEP_ALL_L2;
      N.routed = 0;
      N.ftiles = 1;
      N.ksplit = 1;
      N.kb_total = 0;
      N.kb_per_split = 0;
      N.ntiles = ntiles;
      N.units = M;  // one token row per norm unit
      N.tmB[0] = N.tmB[1] = h->tm_n[bi];
      gf.task[4] = g3.task[0];
      gf.task[4].dep = DEP_OUT_TILE;
      // The output GEMM's K range is [W_up | Ws2]: its Ws2 k-blocks read only the shared
      // L1 output, so they become units of their own, claimed right after the shared L1
      // and run while the routed experts stream, while the W_up k-blocks wait for the norm.
      // Both tasks add partials into the same tiles (one fixed-order reduce).
      {
        GemmTask O = g3.task[0];
        // 256 output features per unit (two 128-row tiles per k-block, one 2 x BN slot)
        if ((H / 128) % 2 == 0) {
          O.pair = 1;
          O.a_rb_up = 1;
          O.a_rb_step = 2;
          O.ftiles = H / 256;
        }
        const int kb_up = L / 64, kb_sh = Is / 64;
        const int tiles = O.ntiles * O.ftiles;
        // The W_up units run after the norm, on the critical path: at most one per SM (a
        // second wave would double the tail).  The Ws2 units take splits of the same size.
        const int ks_want = std::max(1, grid / tiles);
        const int kps = std::max(4, (kb_up + ks_want - 1) / ks_want);
        const int ks_up = (kb_up + kps - 1) / kps, ks_sh = (kb_sh + kps - 1) / kps;
        if (tiles * (ks_up + ks_sh) <= kMaxSplitUnits) {
          GemmTask up = O, sh = O;
          up.kb_lo = 0;
          up.kb_total = kb_up;
          up.kb_per_split = kps;
          up.ksplit = ks_up;
          up.split_base = 0;
          up.ncontrib = ks_up + ks_sh;
          up.units = tiles * ks_up;
          up.dep = DEP_NORM_TILE;
          sh.kb_lo = kb_up;
          sh.kb_total = kb_up + kb_sh;
          sh.kb_per_split = kps;
          sh.ksplit = ks_sh;
          sh.split_base = ks_up;
          sh.ncontrib = ks_up + ks_sh;
          sh.units = tiles * ks_sh;
          sh.dep = DEP_SH_TILE;
          // claim order: S1, R1, OUT(Ws2), R2, NORM, OUT(W_up)
          gf.task[5] = up;
          gf.task[4] = gf.task[3];
          gf.task[3] = gf.task[2];
          gf.task[2] = sh;
          gf.ntasks = 6;
        }
      }
      gf.pf_ptr = reinterpret_cast<const uint8_t*>(h->ws13);
      gf.pf_bytes = 2LL * Is * H * 2;
      gf.l1_done = h->dep_cnt;
      gf.l2_done = h->dep_cnt + h->dep_routed;
      gf.norm_done = gf.l2_done + 1;
      gf.sh_done = gf.norm_done + h->dep_ntiles;
      gf.l1_target = I / 128;
      gf.sh_target = Is / 128;
      gf.l2_ftiles = g2.task[0].ftiles;
      gf.gamma = h->gamma;
      gf.nrm = h->n;
      gf.eps = d.eps;
      KLT_LAUNCH(launch_gemm(gf, BN, grid, s, pdl));
    } else {
      g1.ntasks = 2;
      g1.sched = h->sched + 0;
      g1.stall_after = dbg ? dbg->stall_after_kblocks : 0;
      g1.trace = trace;
      KLT_LAUNCH(launch_gemm(g1, BN, grid, s, pdl));
      g2.ntasks = 1;
      g2.sched = h->sched + 1;
      g2.trace = trace ? trace + trace_launch : nullptr;
      KLT_LAUNCH(launch_gemm(g2, BN, grid, s, pdl));
      NormParams np;
      np.r = h->r;
      np.gamma = h->gamma;
      np.n = h->n;
      np.M = M;
      np.L = L;
      np.eps = d.eps;
      np.zero_r = keep_r ? 0 : 1;
      KLT_LAUNCH(launch_norm(np, s, pdl));
      g3.ntasks = 1;
      g3.sched = h->sched + 2;
      g3.trace = trace ? trace + 2 * trace_launch : nullptr;
      g3.ws = h->ws + ws_task;
      g3.cnt = h->split_cnt + kMaxCounters;
      KLT_LAUNCH(launch_gemm(g3, BN, grid, s, pdl));
    }
  }
#undef KLT_LAUNCH

  // ---- optional copies of routing results and stage outputs
  h->r_dirty = r_left;
  auto cp = [&](void* dst, const void* src, size_t bytes) -> bool {
    return !dst || cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s) == cudaSuccess;
  };
  bool ok = true;
  if (ro) {
    ok &= cp(ro->ids, h->ids, static_cast<size_t>(Mk) * 4);
    ok &= cp(ro->weights, h->wts, static_cast<size_t>(Mk) * 4);
    ok &= cp(ro->cnt, h->cnt, static_cast<size_t>(E) * 4);
    ok &= cp(ro->off, h->off, static_cast<size_t>(E + 1) * 4);
    ok &= cp(ro->gidx, h->gidx, static_cast<size_t>(Mk) * 4);
    ok &= cp(ro->slot, h->slot, static_cast<size_t>(Mk) * 4);
    ok &= cp(ro->pos, h->pos, static_cast<size_t>(Mk) * 4);
  }
  if (dbg) {
    if (mx) ok &= cp(dbg->zsx, h->zsx, static_cast<size_t>(M) * (L / 32));
    if (nv4) ok &= cp(dbg->zsx, h->zsx, static_cast<size_t>(M) * (L / 16));
    if (from_hidden) {
      ok &= cp(dbg->z, h->zp, static_cast<size_t>(M) * L * 2);
      ok &= cp(dbg->logits, h->lgp, static_cast<size_t>(M) * E * 4);
    }
    ok &= cp(dbg->zq, h->zq, static_cast<size_t>(M) * (nv4 ? L / 2 : L));
    ok &= cp(dbg->zs, h->zs, static_cast<size_t>(M) * (L / 128) * 4);
    ok &= cp(dbg->r, h->r, static_cast<size_t>(M) * L * 4);
    ok &= cp(dbg->n, h->n, static_cast<size_t>(M) * L * 2);
    ok &= cp(dbg->a_s, h->a_s, static_cast<size_t>(M) * Is * 2);
    ok &= cp(dbg->aq, h->aq, static_cast<size_t>(Mk) * (nv4 ? I / 2 : I));
    if (dbg->as) {  // stored transposed [I/128, cap] on the device
      const int G = I / 128;
      for (int g = 0; g < G; ++g)
        ok &= cudaMemcpy2DAsync(dbg->as + g, G * sizeof(float),
                                h->asT + static_cast<size_t>(g) * h->cap, sizeof(float),
                                sizeof(float), Mk, cudaMemcpyDeviceToDevice,
                                s) == cudaSuccess;
    }
  }
  return ok ? KLT_OK : KLT_ERR_CUDA;
}

}  // namespace

extern "C" {

int klt_forward(klt_handle* h, const void* x, const void* z, const float* logits, int32_t M,
                void* out, klt_routing* ro, klt_debug* dbg, void* stream) {
  return forward_impl(h, x, z, logits, M, out, ro, dbg, stream, false);
}

int klt_forward_hidden(klt_handle* h, const void* x, int32_t M, void* out, klt_routing* ro,
                       klt_debug* dbg, void* stream) {
  return forward_impl(h, x, nullptr, nullptr, M, out, ro, dbg, stream, true);
}

int klt_status(klt_handle* h) {
  if (!h) return KLT_ERR_INVALID_ARG;
  int e = 0;
  if (cudaMemcpy(&e, h->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return KLT_ERR_CUDA;
  if (e) h->r_dirty = true;  // a stopped forward may have left partial sums in r
  return e ? KLT_ERR_DEVICE_TIMEOUT : KLT_OK;
}

int klt_destroy(klt_handle* h) {
  if (!h) return KLT_OK;
  cudaDeviceSynchronize();
  free_all(h);
  delete h;
  return KLT_OK;
}

}  // extern "C"
