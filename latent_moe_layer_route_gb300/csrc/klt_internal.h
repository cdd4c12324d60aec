// Host/device shared definitions of the latent-MoE tail library: kernel parameter blocks
// and the launchers each kernel file exports to the host API.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace klt {

// ------------------------------------------------------------------ routing kernels
// Block-scaled routed formats (the tensor core applies the scales): MXFP8 (e4m3 with an
// UE8M0 scale per 32) and NVFP4 weights and activations (e2m1 with an e4m3 scale per 16).
enum BlockScale : int { BS_NONE = 0, BS_MX8 = 1, BS_NV4 = 2 };

struct RouteParams {
  const float* logits;     // [M, E]
  const __nv_bfloat16* z;  // [M, L]
  int32_t* ids;            // [M, k]
  float* wts;              // [M, k]
  uint8_t* zq;             // [M, L]
  float* zs;               // [M, L/128]
  float* r;                // [M, L] fp32 combine buffer (zeroed by the previous norm)
  int* sched;              // per-launch tile counters, zeroed here
  int nsched;
  int* zero_buf;           // dependency counters of the fused launch, zeroed here
  int zero_n;
  int M, E, k, L;
  int bs;                  // activation format: BS_NONE (fp32 scale per 128 into zs),
                           // BS_MX8 (UE8M0 byte per 32 columns into zsx) or BS_NV4 (e2m1
                           // codes packed two per byte into zq, e4m3 byte per 16 into zsx)
  uint8_t* zsx;            // [M, L/32] or [M, L/16]
};

struct PermParams {
  const int32_t* ids;  // [M*k]
  int* hist;           // [nblocks, E] per-block expert counts
  int32_t* cnt;        // [E]
  int32_t* off;        // [E+1]
  int32_t* tile_off;   // [E+1] prefix of ceil(cnt/BN)
  int32_t* gidx;       // [cap]
  int32_t* slot;       // [cap]
  int32_t* pos;        // [M*k]
  const uint8_t* zq;   // [M, L]
  const float* zs;     // [M, L/128]
  uint8_t* zq_perm;    // [cap, L]
  __nv_bfloat16* zqb_perm;  // [cap, L] exact bf16 images of the codes (bf16-operand layers)
  float* zsT;          // [L/128, cap]
  const float* wts;    // [M*k] routing weights by pair i
  float* wperm;        // [cap] routing weight of pair p
  int M, E, k, L, cap, bn, nblocks;
  // Block-scaled layers: the gathered token scale bytes as 512-byte tiles, one per
  // (routed tile of bn = 128 pairs, 4 consecutive scale bytes of a row), laid out for
  // tcgen05.cp: byte r%32*16 + 4*(r/32) + j = scale 4a + j of tile row r in tile a (rows
  // past the tile: scale 1).  sf_group columns per scale byte: 32 (MX, a tile per
  // 128-column k-block) or 16 (NVFP4 activations, a tile per 64 columns).
  const uint8_t* zsx;  // [M, L/sf_group]
  uint8_t* zsf_t;      // [tile capacity, L/(4 sf_group), 512]
  int sf_tiles;        // tile capacity (grid bound; tile_off[E] of the batch is <= it)
  int sf_group;
  int zrow;            // bytes per quantised latent row: L (e4m3) or L/2 (packed e2m1)
};

struct NormParams {
  float* r;                    // [M, L]
  const __nv_bfloat16* gamma;  // [L]
  __nv_bfloat16* n;            // [M, L]
  int M, L;
  float eps;
  int zero_r;  // zero each row of r after normalising it (ready for the next forward)
};

// ------------------------------------------------------------------ tile GEMM engine
enum TaskKind : int {
  TASK_NONE = 0,
  TASK_SHARED_L1 = 1,  // bf16 x . Ws13^T, gate/up pair -> SwiGLU -> a_s (bf16)
  TASK_ROUTED_L1 = 2,  // fp8 zq_perm . W13_e^T, pair, per-128-K promotion -> SwiGLU ->
                       // per-128 e4m3 quantisation -> aq, asT
  TASK_ROUTED_L2 = 3,  // fp8 aq . W2_e^T, promotion -> r[gidx] += w * y (fp32 atomics)
  TASK_OUT = 4,        // bf16 [n | a_s] . [W_up | Ws2]^T -> out (bf16, one rounding)
  TASK_NORM = 5,       // RMSNorm of a token tile of r -> n (epilogue warps, no MMA)
  TASK_PROJ = 6        // bf16 x . [W_lat | W_gate]^T -> latent input z (bf16, rows < L)
                       // and router logits (fp32, rows L .. L+E-1); the step before the tail
};

// Dependency of a unit in the fused launch, checked by the producer before it publishes
// the unit (and before it copies the token operand).
enum DepKind : int {
  DEP_NONE = 0,
  DEP_L1_TILE = 1,   // routed L2 unit: all L1 units of its routed token tile are done
  DEP_ALL_L2 = 2,    // norm unit: every routed L2 unit is done
  DEP_OUT_TILE = 3,  // output unit: norm and shared L1 of its token tile are done
  DEP_SH_TILE = 4,   // output unit over the shared down-projection's k-blocks only: the
                     // shared L1 tiles of its token tile are done
  DEP_NORM_TILE = 5  // output unit over the up-projection's k-blocks only: the norm rows
                     // of its token tile are done
};

struct GemmTask {
  CUtensorMap tmB[2];  // token operand maps (BN-row boxes); [1] used past kb_split0
  const uint8_t* a_ptr[2];  // weight operands, pre-swizzled tile-major (16 KB per tile)
  int kind;
  int fp8;             // operands e4m3 (kind::f8f6f4, 128 elements per k-block) or bf16
                       // (kind::f16, 64 elements per k-block)
  int kpg;             // k-blocks per promotion group (0: accumulate the unit in TMEM)
  int routed;          // units come from the device tile list (tile_off/off)
  int ftiles;          // 128-row output tiles (gate/up pairs for L1 kinds)
  int kb_total;        // k-blocks of 128 bytes per row (end of this task's k range)
  int kb_split0;       // k-blocks served by map pair 0
  int kb_lo;           // first k-block of this task's k range (0 unless a tile's K range
                       // is shared out between two tasks)
  int ksplit;          // k splits of [kb_lo, kb_total); >1 => partials + last-arriver reduce
  int kb_per_split;
  int split_base;      // index of this task's first split among its tile's contributions
  int ncontrib;        // contributions per tile over all tasks sharing it (0: ksplit)
  int pair;            // feature-major engine: each unit reads two 128-row weight tiles per
                       // k-block into one accumulator slot of 2 x BN columns (gate and up
                       // of the L1 kinds, or two consecutive row blocks of W2)
  int a_rb_up;         // 128-row blocks from a unit's first weight tile to its second (pairs)
  int a_rb_step;       // 128-row blocks per output tile index (2 for paired W2 units, else 1)
  int a_rb_expert;     // routed: 128-row blocks per expert
  int a_kb[2];         // k-blocks per 128-row block of a_ptr[0], a_ptr[1]
  int ntiles;          // non-routed: token tiles
  int dual;            // token-major engine, non-promoted: a unit covers two token tiles
                       // that share its weight tiles (units = ceil(ntiles / 2) * ftiles)
  int units;           // non-routed: ntiles * ftiles * ksplit
  int dep;             // DepKind of this task's units
  // Block-scaled units (token-major engine): scale tiles of 512 bytes in the tcgen05.cp
  // layout, the weights' per 128-row block like their data tiles, the tokens' per routed
  // tile, in K order (MX: one tile per k-block; NVFP4: four, one per 64-wide MMA);
  // null for other tasks
  const uint8_t* a_sf;
  const uint8_t* t_sf;
  const float* a_g;    // NVFP4 units: the weights' fp32 per-matrix scale [E] (epilogue)
  int ws_tile_base;    // first arrival counter of this task (tile ids start here)
  long long ws_off;    // float offset of this task's partials in the workspace
  int streamk;         // 1: static stream-K partition of ntiles*ftiles*kb_total k-blocks
                       //    over sk_grid CTAs (non-routed, bf16, sole task of its launch)
  int sk_grid;
  long long sk_total;
};

constexpr int kMaxTasks = 6;

struct GemmParams {
  GemmTask task[kMaxTasks];
  int ntasks;
  int M;                       // tokens of this forward
  int E, L, I, Is, H, cap;     // cap = max_tokens * topk (rows of the permuted buffers)
  const int32_t* tile_off;     // [E+1]
  const int32_t* off;          // [E+1]
  const int32_t* gidx;         // [cap]
  const float* wperm;          // [cap] routing weight of pair p
  const float* zsT;            // [L/128, cap]
  const float* w13_s;          // [E, 2I/128, L/128]
  const float* w2_s;           // [E, L/128, I/128]
  uint8_t* aq;                 // [cap, I]
  __nv_bfloat16* aqb;          // [cap, I] exact bf16 images of aq (bf16-operand layers) or null
  float* asT;                  // [I/128, cap]
  float* r;                    // [M, L]
  // deterministic combine (null yw: the routed L2 units add into r): the routed L2 units
  // store w * y per permuted pair into yw and the norm sums a token's topk slots in order
  float* yw;                   // [cap, L] or null
  const int32_t* pos;          // [M, topk] permuted pair of (token, choice)
  int topk;
  __nv_bfloat16* a_s;          // [max_tokens, Is]
  __nv_bfloat16* out;          // [M, H]
  float* ws;                   // split-K partials
  int* cnt;                    // split-K arrival counters (zero between uses)
  int* sched;                  // this launch's dynamic tile counter (zeroed by routing)
  int* err;                    // sticky device error word
  long long timeout;           // SM cycles per bounded wait
  int stall_after;             // test hook (0 = off)
  // fused launch: dependency counters (zeroed by the routing kernel) and the norm step
  int* l1_done;                // [routed tiles] L1 units done per routed token tile
  int* l2_done;                // routed L2 units done
  int* norm_done;              // [token tiles] norm units done
  int* sh_done;                // [token tiles] shared L1 tiles finalised
  int l1_target;               // L1 units per routed token tile (I/128)
  int sh_target;               // shared L1 tiles per token tile (Is/128)
  int l2_ftiles;               // routed L2 units per routed token tile (L/128)
  const __nv_bfloat16* gamma;  // [L]
  __nv_bfloat16* nrm;          // [max_tokens, L]
  float eps;
  int w_stages;                // token-major engine: stage ring depth (4 x 48 KB or 3 x 64 KB)
  int w_stage_bytes;           //   and stage size (64 KB when units carry two token tiles)
  // routing-independent weights prefetched into L2 before the launch waits for the
  // preceding kernel (16-byte aligned, a multiple of 16 bytes; null/0: none)
  const uint8_t* pf_ptr;
  long long pf_bytes;
  int bs;                      // token-major engine, block-scaled layer (BlockScale):
                               // block-scaled routed units (one accumulator slot; the scale
                               // ring takes the other half of TMEM) and the routed L1
                               // epilogue requantises (MX: per 32 with power-of-two scales;
                               // NVFP4: per 16 to e2m1 with e4m3 scales) into aq and the
  uint8_t* asf_t;              //   token scale tiles of the L2 [tiles, I/(4 group), 512]
  __nv_bfloat16* zp;           // projection outputs: latent input [M, L]
  float* lgp;                  //   and router logits [M, E]
  long long* trace;            // optional timestamp trace (this launch's region)
  int trace_n;                 // entries per (CTA, role)
  int zero_r;                  // norm units zero each row of r once it is normalised, so
                               // the next forward's routed L2 units add into zeros
  // token-major output GEMM split in K (few token tiles): the splits add into out_acc and
  // the last of a tile rounds it into out, then zeroes its rows and its counter
  float* out_acc;              // [kWideSplitMaxTiles * 128, H] fp32, zero between uses
  int* out_cnt;                // [kWideSplitMaxTiles * H / 256] arrivals, zero between uses
};

// Launchers (return cudaError_t of the launch).
cudaError_t launch_route(const RouteParams& p, cudaStream_t s, bool pdl);
cudaError_t launch_perm_hist(const PermParams& p, cudaStream_t s, bool pdl);
cudaError_t launch_perm_scatter(const PermParams& p, cudaStream_t s, bool pdl);
cudaError_t launch_perm_gather(const PermParams& p, cudaStream_t s, bool pdl);
// route + scatter + gather in one launch; needs M·k <= SMALL_PAIRS and e4m3 activations
cudaError_t launch_route_small(const RouteParams& rp, const PermParams& p, cudaStream_t s,
                               bool pdl);
cudaError_t launch_norm(const NormParams& p, cudaStream_t s, bool pdl);
// Row-major [rows, row_bytes] -> 128-row x 128-byte tiles, tile (rb, kb) at
// ((rb * row_bytes/128) + kb) * 16384 bytes (rows % 128 == 0, row_bytes % 128 == 0), each
// tile stored in the 128-byte-swizzled K-major image the tensor core reads from shared
// memory: 16-byte chunk c of row r at r * 128 + (c ^ (r % 8)) * 16.
// NVFP4 [rows, K/2] packed e2m1 + e4m3 scales [rows, K/16] -> exact bf16 values
// e2m1 * scale (the per-matrix fp32 scale is applied later) in the same swizzled tile-major
// image as launch_tile_relayout for a bf16 matrix [rows, K].
cudaError_t launch_nvfp4_expand(const uint8_t* packed, const uint8_t* sb, void* dst,
                                long long rows, long long K, cudaStream_t s);
// dst[e * per + i] = g[e] for i < per (per-128-block promotion scales of NVFP4 layers).
cudaError_t launch_fill_expert_scale(const float* g, float* dst, int E, long long per,
                                     cudaStream_t s);
cudaError_t launch_tile_relayout(const void* src, void* dst, long long rows, long long row_bytes,
                                 cudaStream_t s);
// Scale bytes [rows, nsc] (rows % 128 == 0, nsc % 4 == 0) -> 512-byte tiles per (128-row
// block rb, group of 4 scale bytes a) at (rb * nsc/4 + a) * 512, byte (r%32)*16 +
// 4*((r%128)/32) + j = scale 4a + j of row r (the tcgen05.cp 32x128b layout).
cudaError_t launch_sf_relayout(const uint8_t* src, uint8_t* dst, long long rows, long long nsc,
                               cudaStream_t s);
// bn in {16, 128}; grid = persistent CTAs.
cudaError_t launch_gemm(const GemmParams& p, int bn, int grid, cudaStream_t s, bool pdl);
int gemm_smem_bytes(int bn);
// The feature-major engine hands registers from its control warps to its epilogue warps at
// run time: every instantiation must launch with the register count that was planned.
bool gemm_regs_ok();
// Token-major engine (128-token x 256-feature units, one persistent launch of the five
// fused tasks with 128-token tiles).  Its epilogue warps take registers from the control
// warps at run time, which needs the kernel to launch with exactly the register count it
// was built for: wide_regs_ok(wide_kernel_regs()) must hold before launch_wide is used.
// Token-major engine: RMSNorm rows per norm unit (one per epilogue warp).
constexpr int kWideNormRows = 8;
// Token-major output GEMM: split in K for batches of at most this many 128-token tiles.
constexpr int kWideSplitMaxTiles = 2;
cudaError_t launch_wide(const GemmParams& p, int grid, cudaStream_t s, bool pdl);
int wide_kernel_regs();
bool wide_regs_ok(int regs);

constexpr int PERM_BLOCK = 1024;  // pairs per permutation block
constexpr int ROUTE_WARPS = 8;    // warps per routing block
constexpr int ROUTE_QG = 4;       // 128-column latent groups quantised per routing warp
constexpr int SMALL_PAIRS = 256;  // most pairs the one-launch routing takes
constexpr int SMALL_THREADS = 512;  // threads per block of the one-launch routing
constexpr int MAX_TOPK = 32;
constexpr int MAX_E = 256;
constexpr int MAX_KB = 32;       // routed K blocks of 128 per unit (L, I <= 4096)

}  // namespace klt
