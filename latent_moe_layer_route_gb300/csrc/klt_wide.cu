// Token-major tile engine for prefill batches: one persistent launch runs the routed L1
// (SwiGLU + per-token e4m3 requantisation), the shared-expert L1, the routed L2 with the
// weighted scatter-combine, the RMSNorm and the output GEMM, like the decode engine, but
// every unit is a 128-token x 256-feature tile:
//
//   D[token, feature] = sum_k A[token, k] * B[feature, k]      (tcgen05.mma M=128, N=256)
//
// A is the token tile (TMA, 128 rows x 128 bytes per k-block) and B is two pre-swizzled
// 128-row weight tiles placed back to back (gate and up of an L1 unit, or two consecutive
// row blocks of L2 / output weights).  With 256 features per MMA the tensor pipe, not the
// single issuing thread, sets the pace, and each staged byte feeds twice the MMA work of a
// 128-feature tile.  From 16 token tiles on, the BF16 tasks (shared L1, output GEMM) run
// dual units: two token tiles share each staged weight tile and fill both TMEM slots.
//
// Warp roles (3 warpgroups): warp 0 = TMA producer, warp 1 = MMA issuer, warp 2 = unit
// completion signaller, warp 3 idle, warps 4-11 = epilogue.  The control warpgroup hands registers to the epilogue
// warpgroups (setmaxnreg) so each epilogue thread can hold its 128 fp32 accumulators of
// one token across the per-128-K promotion of block-scaled FP8 (or NVFP4) products.
//
// Epilogue thread (warp w, lane l): token row (w % 4) * 32 + l of the tile (its TMEM lane)
// and column half h = (w - 4) / 4: for gate/up units gate columns [64h, 64h+64) and up
// columns [128+64h, 128+64h+64), otherwise columns [128h, 128h+128).
#include "klt_device.cuh"
#include "klt_internal.h"

namespace klt {

namespace {

struct W {
  static constexpr int TM = 128;  // tokens per tile: MMA M, TMEM lanes
  static constexpr int TN = 256;  // features per unit: MMA N, TMEM columns per slot
  static constexpr int EPI_WARPS = 8;
  static constexpr int FIRST_EPI_WARP = 4;
  static constexpr int THREADS = 12 * 32;
  static constexpr int EPI_THREADS = EPI_WARPS * 32;
  static constexpr int NORM_ROWS = kWideNormRows;  // one token row per epilogue warp
  static_assert(NORM_ROWS == EPI_WARPS && TM % NORM_ROWS == 0, "norm rows per unit");
  static constexpr int W_TILE = 128 * 128;  // one pre-swizzled weight tile
  static constexpr int T_TILE = TM * 128;   // token tile of one k-block
  // The stage ring is 192 KB, either 4 stages of two weight tiles + one token tile or 3
  // stages with room for a second token tile (dual units of the BF16 tasks); the launch
  // chooses (GemmParams::w_stages, w_stage_bytes).  Barriers are sized for the deeper ring.
  static constexpr int STAGE_BYTES = 2 * W_TILE + T_TILE;
  static constexpr int STAGES = 4;
  static constexpr int DUAL_STAGE_BYTES = 2 * W_TILE + 2 * T_TILE;
  static constexpr int DUAL_STAGES = 3;
  static_assert(STAGES * STAGE_BYTES == DUAL_STAGES * DUAL_STAGE_BYTES, "one ring size");
  static constexpr int TMEM_COLS = 512;
  static constexpr int NACC = TMEM_COLS / TN;  // accumulator slots (MX launches use one)
  static constexpr int SF_STAGE = 3 * 512;     // MX scale tiles per stage
  static constexpr int SF_COLS = 12;           // TMEM columns of one stage's scales
  static_assert(TN + STAGES * SF_COLS <= TMEM_COLS, "MX scale ring beside one slot");
  // NVFP4 (e2m1 x e2m1) routed units: each stage also carries their scale tiles after the
  // token tile (4 x 512 bytes for the 128 token rows and 8 x 512 for the 256 weight rows,
  // one tile per 64-wide MMA), in a ring of 3 stages; a stage's tiles take 48 TMEM
  // columns beside the single accumulator slot.
  static constexpr int NV4_SF_BYTES = 12 * 512;
  static constexpr int NV4_STAGE_BYTES = STAGE_BYTES + NV4_SF_BYTES;
  static constexpr int NV4_STAGES = 3;
  static constexpr int NV4_SF_COLS = 48;
  static_assert(NV4_STAGES * NV4_STAGE_BYTES <= STAGES * STAGE_BYTES, "NVFP4 ring fits");
  static_assert(NV4_STAGE_BYTES % 1024 == 0, "stage alignment of the swizzled tiles");
  static_assert(TN + NV4_STAGES * NV4_SF_COLS <= TMEM_COLS, "NVFP4 scale ring beside one slot");
  static constexpr int US = 8;
  static constexpr int SIG = 8;             // completion-signal ring (epilogue -> signaller)
  static constexpr int SIGNAL_WARP = 2;     // control warp that publishes unit completions
  // Registers: 384 threads launch with 168 each (3 warps share a scheduler); the control
  // warpgroup drops to 72 and the two epilogue warpgroups rise to 216, exactly the
  // registers released (72 keeps the producer's scale-tile paths and the MMA issuer's
  // block-scaled loop free of spills).
  static constexpr int LAUNCH_REGS = 168;
  static constexpr int REGS_CTRL = 72;
  static constexpr int REGS_EPI = 216;
  static_assert(4 * (LAUNCH_REGS - REGS_CTRL) >= 8 * (REGS_EPI - LAUNCH_REGS),
                "register hand-over must balance");
  static_assert(NACC == 2, "two accumulator slots");
};

struct WUnit {
  int task;   // -1: no more work
  int e;      // routed expert
  int row0;   // first token row of the tile
  int rows;   // valid token rows
  int ftile;  // output feature tile (128 SwiGLU outputs for gate/up kinds, else 256)
  int rb0, rb1;  // weight row blocks staged as B rows [0, 128) and [128, 256)
  int dep_idx;  // routed token tile (routed kinds) or token tile (others)
  int dual;     // 1: a second token tile follows (rows from row0 + TM, token tile dep_idx + 1)
  int kb0, kb1;  // k-blocks [kb0, kb1) of the unit (a k-split output unit: one split)
};

// Combine staging: per warp 32 tokens x 16 features (fp32), each row's four 16-byte quads
// stored at quad position j ^ ((row >> 1) & 3), so that both the row-wise 16-byte stores
// of 8 lanes and the quad-wise 16-byte loads of 8 lanes touch 32 different banks.
constexpr int STG_LD = 16;
__device__ __forceinline__ int stg_quad(int row, int j) { return row * STG_LD + 4 * (j ^ ((row >> 1) & 3)); }

struct WSmem {
  uint8_t* stages;
  uint64_t *full, *empty, *tfull, *tempty, *ufull, *uempty, *sfull, *sempty, *drain;
  int** sptr;  // [SIG] counter each completion signal increments (null: end of work)
  WUnit* ring;
  uint32_t* tmem_holder;
  int* abort_flag;
  int* split_last;  // k-split output units: set when this CTA's split was a tile's last
  float* amax;  // [2 unit parities][2 column halves][TM]
  float* stg;   // [EPI_WARPS][32 tokens][STG_LD] per-warp transpose staging of the combine
                // (16-byte aligned)
  uint8_t* sf;  // [STAGES][SF_STAGE] MX scale tiles of each stage: tokens, weight rows
                // 0-127, weight rows 128-255 (512 bytes each, 16-byte aligned)

  static constexpr int BAR_BYTES =
      8 * (2 * W::STAGES + 2 * W::NACC + 2 * W::US + 2 * W::SIG + 1) + 8 * W::SIG;
  static constexpr int bytes() {
    return W::STAGES * W::STAGE_BYTES + BAR_BYTES + W::US * (int)sizeof(WUnit) + 64 +
           4 * W::TM * 4 + W::EPI_WARPS * 32 * STG_LD * 4 + W::STAGES * W::SF_STAGE +
           16 + 1024 /* alignment slack */;
  }
  __device__ explicit WSmem(uint8_t* raw) {
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023));
    stages = base;
    uint64_t* b = reinterpret_cast<uint64_t*>(base + W::STAGES * W::STAGE_BYTES);
    full = b;
    empty = full + W::STAGES;
    tfull = empty + W::STAGES;
    tempty = tfull + W::NACC;
    ufull = tempty + W::NACC;
    uempty = ufull + W::US;
    sfull = uempty + W::US;
    sempty = sfull + W::SIG;
    drain = sempty + W::SIG;
    sptr = reinterpret_cast<int**>(drain + 1);
    ring = reinterpret_cast<WUnit*>(sptr + W::SIG);
    tmem_holder = reinterpret_cast<uint32_t*>(ring + W::US);
    abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
    split_last = reinterpret_cast<int*>(tmem_holder + 2);
    amax = reinterpret_cast<float*>(tmem_holder + 16);
    stg = reinterpret_cast<float*>(
        (reinterpret_cast<uintptr_t>(amax + 4 * W::TM) + 15) & ~static_cast<uintptr_t>(15));
    sf = reinterpret_cast<uint8_t*>(stg + W::EPI_WARPS * 32 * STG_LD);
  }
};

__device__ __forceinline__ void trace_mark(const GemmParams& p, int role, int i) {
  if (p.trace != nullptr && i < p.trace_n)
    p.trace[(static_cast<long long>(blockIdx.x) * 4 + role) * p.trace_n + i] = global_ns();
}

__device__ __forceinline__ bool is_pair(int kind) {
  return kind == TASK_SHARED_L1 || kind == TASK_ROUTED_L1;
}

// Unit u of the launch, tasks in order.  Routed units: token tile t of the device tile
// list (128 tokens of one expert), feature tile ft, t-major so an expert's token tiles
// read its weights close together in time.
__device__ WUnit w_decode(const GemmParams& p, const int* s_tile_off, const int* s_off, int u) {
  WUnit info;
  info.task = -1;
  for (int ti = 0; ti < p.ntasks; ++ti) {
    const GemmTask& T = p.task[ti];
    const bool pair = is_pair(T.kind);
    if (T.routed) {
      const int units = s_tile_off[p.E] * T.ftiles;
      if (u < units) {
        const int t = u / T.ftiles;
        const int ft = u - t * T.ftiles;
        int lo = 0, hi = p.E - 1;  // largest e with tile_off[e] <= t
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (s_tile_off[mid] <= t) lo = mid; else hi = mid - 1;
        }
        info.task = ti;
        info.e = lo;
        info.row0 = s_off[lo] + (t - s_tile_off[lo]) * W::TM;
        info.rows = min(W::TM, s_off[lo + 1] - info.row0);
        info.ftile = ft;
        info.rb0 = lo * T.a_rb_expert + (pair ? ft : 2 * ft);
        info.rb1 = pair ? info.rb0 + T.a_rb_up : info.rb0 + 1;
        info.dep_idx = t;
        info.dual = 0;
        info.kb0 = 0;
        info.kb1 = T.kb_total;
        return info;
      }
      u -= units;
    } else {
      if (u < T.units) {
        info.task = ti;
        info.e = 0;
        info.dual = 0;
        info.kb0 = 0;
        info.kb1 = T.kb_total;
        if (T.kind == TASK_NORM) {  // NORM_ROWS token rows, all in one token tile
          info.row0 = u * W::NORM_ROWS;
          info.rows = min(W::NORM_ROWS, p.M - info.row0);
          info.ftile = 0;
          info.rb0 = info.rb1 = 0;
          info.dep_idx = info.row0 / W::TM;
        } else {
          // feature-tile major: every token tile of a weight tile runs close together in
          // time, so each weight tile is read from DRAM once and stays hot in L2; a k-split
          // task (single token tiles) has its splits innermost
          const int ks = T.ksplit;
          const int per_ft = (T.dual ? (T.ntiles + 1) / 2 : T.ntiles) * ks;
          const int ft = u / per_ft;
          const int js = u - ft * per_ft;
          const int j = js / ks;
          if (ks > 1) {
            info.kb0 = (js - j * ks) * T.kb_per_split;
            info.kb1 = min(T.kb_total, info.kb0 + T.kb_per_split);
          }
          const int nt = T.dual ? 2 * j : j;
          info.row0 = nt * W::TM;
          info.rows = min(W::TM, p.M - info.row0);
          info.ftile = ft;
          info.rb0 = pair ? ft : 2 * ft;
          info.rb1 = pair ? info.rb0 + T.a_rb_up : info.rb0 + 1;
          info.dep_idx = nt;
          info.dual = T.dual && nt + 1 < T.ntiles;
        }
        return info;
      }
      u -= T.units;
    }
  }
  return info;
}

// Bounded wait until the unit's inputs produced by other units of this launch are complete
// (acquire loads pairing with the producers' release adds; the proxy fence orders the
// acquired data before this thread's TMA reads of it).
__device__ bool w_wait_dependency(const GemmParams& p, int dep, int idx, const int* s_tile_off,
                                  volatile int* abort_flag) {
  if (dep == DEP_NONE) return true;
  const long long t0 = clock64();
  for (;;) {
    bool ready;
    if (dep == DEP_L1_TILE) {
      ready = ld_acquire_gpu(p.l1_done + idx) >= p.l1_target;
    } else if (dep == DEP_ALL_L2) {
      ready = ld_acquire_gpu(p.l2_done) >= s_tile_off[p.E] * p.l2_ftiles;
    } else {
      ready = ld_acquire_gpu(p.norm_done + idx) >=
                  (min(W::TM, p.M - idx * W::TM) + W::NORM_ROWS - 1) / W::NORM_ROWS &&
              ld_acquire_gpu(p.sh_done + idx) >= p.sh_target;
    }
    if (ready) break;
    if (*abort_flag) return false;
    if (clock64() - t0 > p.timeout) {
      *abort_flag = 1;
      atomicOr(p.err, DEV_ERR_TIMEOUT);
      return false;
    }
    __nanosleep(100);
  }
  fence_proxy_async_global();
  return true;
}

// ------------------------------------------------------------------ producer (1 thread)
// BS: the launch carries block-scaled routed units of that format (their own kernel
// instantiation, so the other launches keep their code and registers unchanged).
template <int BS>
__device__ void w_producer(const GemmParams& p, WSmem& sm, const int* s_tile_off,
                           const int* s_off, int u0) {
  // weights are re-read by every token tile of their expert, tokens by every feature tile
  const uint64_t pol = policy_evict_normal();
  const uint64_t pol_w = policy_evict_last();
  const int nst = p.w_stages, sbytes = p.w_stage_bytes;
  int stage = 0, us = 0;
  uint32_t phase = 0, uphase = 0;
  long long issued = 0;
  int published = 0;
  int dummy_abort = 0;
  bool stalled = false;
  int u = u0;  // first unit, claimed by the caller
  for (;;) {
    const WUnit info = w_decode(p, s_tile_off, s_off, u);
    // claim the next unit now so the counter round trip overlaps this unit's copies
    if (info.task >= 0) u = atomicAdd(p.sched, 1);
    if (info.task < 0) {
      if (mbar_wait(&sm.uempty[us], uphase ^ 1, sm.abort_flag, p.err, p.timeout)) {
        sm.ring[us] = info;
        mbar_arrive(&sm.ufull[us]);
      }
      break;
    }
    const GemmTask& T = p.task[info.task];
    const int elems_per_kb = T.fp8 ? 128 : 64;
    const bool mxu = BS == BS_MX8 && T.a_sf != nullptr;  // block-scaled: scale tiles ride along
    const bool nvu = BS == BS_NV4 && T.a_sf != nullptr;
    auto issue_w = [&](int kb, uint8_t* st) {
      const int m = kb < T.kb_split0 ? 0 : 1;
      const int kk = m ? kb - T.kb_split0 : kb;
      const uint8_t* a = T.a_ptr[m];
      const size_t akb = static_cast<size_t>(T.a_kb[m]);
      bulk_load(st, a + (static_cast<size_t>(info.rb0) * akb + kk) * W::W_TILE, W::W_TILE,
                &sm.full[stage], pol_w);
      bulk_load(st + W::W_TILE, a + (static_cast<size_t>(info.rb1) * akb + kk) * W::W_TILE,
                W::W_TILE, &sm.full[stage], pol_w);
      if (mxu) {
        uint8_t* sf = sm.sf + stage * W::SF_STAGE;
        bulk_load(sf + 512, T.a_sf + (static_cast<size_t>(info.rb0) * akb + kk) * 512, 512,
                  &sm.full[stage], pol_w);
        bulk_load(sf + 1024, T.a_sf + (static_cast<size_t>(info.rb1) * akb + kk) * 512, 512,
                  &sm.full[stage], pol_w);
      }
      if (nvu) {  // the four 512-byte tiles of each weight row block for this k-block
        uint8_t* sf = st + 2 * W::W_TILE + W::T_TILE;
        bulk_load(sf + 2048, T.a_sf + (static_cast<size_t>(info.rb0) * akb + kk) * 2048, 2048,
                  &sm.full[stage], pol_w);
        bulk_load(sf + 4096, T.a_sf + (static_cast<size_t>(info.rb1) * akb + kk) * 2048, 2048,
                  &sm.full[stage], pol_w);
      }
    };
    auto issue_t = [&](int kb, uint8_t* st, uint64_t* bar, int stg_idx) {
      const int m = kb < T.kb_split0 ? 0 : 1;
      const int kk = m ? kb - T.kb_split0 : kb;
      tma_load_2d(st + 2 * W::W_TILE, &T.tmB[m], bar, kk * elems_per_kb, info.row0, pol);
      if (info.dual)
        tma_load_2d(st + 2 * W::W_TILE + W::T_TILE, &T.tmB[m], bar, kk * elems_per_kb,
                    info.row0 + W::TM, pol);
      if (mxu)  // this routed tile's token scales for the k-block
        bulk_load(sm.sf + stg_idx * W::SF_STAGE,
                  T.t_sf + (static_cast<size_t>(info.dep_idx) * T.kb_total + kk) * 512, 512, bar,
                  pol);
      if (nvu)  // the routed tile's four token scale tiles of the k-block
        bulk_load(st + 2 * W::W_TILE + W::T_TILE,
                  T.t_sf + (static_cast<size_t>(info.dep_idx) * T.kb_total + kk) * 2048, 2048,
                  bar, pol);
    };
    const uint32_t stage_tx = 2 * W::W_TILE +
                              (info.dual ? 2 : 1) * static_cast<uint32_t>(W::T_TILE) +
                              (mxu ? W::SF_STAGE : 0) + (nvu ? W::NV4_SF_BYTES : 0);
    // (block-scaled launches run routed units only, which are never split in K)
    const int kb_end = BS != BS_NONE ? T.kb_total : info.kb1;
    const int kb_first = BS != BS_NONE ? 0 : info.kb0;
    int kb = kb_first;
    if (T.dep != DEP_NONE) {
      // Stream the unit's weight tiles into the stages that are free now, then wait for
      // the token operand's producers, then copy the token tiles of those stages.
      // the early stages are consecutive ring slots holding k-blocks kb0, kb0 + 1, ...
      const int st0 = stage;
      int npre = 0;
      while (kb < kb_end && npre < nst) {
        if (p.stall_after > 0 && issued >= p.stall_after) break;
        if (!mbar_try_wait(&sm.empty[stage], phase ^ 1)) break;
        uint8_t* st = sm.stages + stage * sbytes;
        mbar_arrive_expect_tx(&sm.full[stage], stage_tx);
        issue_w(kb, st);
        ++npre;
        trace_mark(p, 0, static_cast<int>(issued));
        ++issued;
        if (++stage == nst) { stage = 0; phase ^= 1; }
        ++kb;
      }
      if (!w_wait_dependency(p, T.dep, info.dep_idx, s_tile_off, sm.abort_flag)) break;
      if (info.dual &&
          !w_wait_dependency(p, T.dep, info.dep_idx + 1, s_tile_off, sm.abort_flag))
        break;
      for (int i = 0, s = st0; i < npre; ++i) {
        issue_t(kb_first + i, sm.stages + s * sbytes, &sm.full[s], s);
        if (++s == nst) s = 0;
      }
    }
    if (!mbar_wait(&sm.uempty[us], uphase ^ 1, sm.abort_flag, p.err, p.timeout)) break;
    sm.ring[us] = info;
    mbar_arrive(&sm.ufull[us]);
    if (++us == W::US) { us = 0; uphase ^= 1; }
    if (p.trace != nullptr && published < p.trace_n) {  // unit publish time and task
      p.trace[(static_cast<long long>(blockIdx.x) * 4 + 1) * p.trace_n + published] = global_ns();
      p.trace[(static_cast<long long>(blockIdx.x) * 4 + 3) * p.trace_n + published] =
          info.task + 1;
    }
    ++published;
    for (; kb < kb_end; ++kb) {
      if (p.stall_after > 0 && issued >= p.stall_after) { stalled = true; break; }
      if (!mbar_wait_spin(&sm.empty[stage], phase ^ 1, sm.abort_flag, p.err, p.timeout)) {
        stalled = true;
        break;
      }
      uint8_t* st = sm.stages + stage * sbytes;
      mbar_arrive_expect_tx(&sm.full[stage], stage_tx);
      issue_w(kb, st);
      issue_t(kb, st, &sm.full[stage], stage);
      trace_mark(p, 0, static_cast<int>(issued));
      ++issued;
      if (++stage == nst) { stage = 0; phase ^= 1; }
    }
    if (stalled) break;
  }
  // Drain: wait (bounded, ignoring the abort flag) for this thread's last copies, so no
  // TMA write into shared memory outlives the CTA.
  const long long first = issued > nst ? issued - nst : 0;
  for (long long i = first; i < issued; ++i) {
    const int s = static_cast<int>(i % nst);
    const uint32_t par = static_cast<uint32_t>((i / nst) & 1);
    mbar_wait(&sm.full[s], par, &dummy_abort, p.err, p.timeout);
  }
}

// ------------------------------------------------------------------ MMA issuer (1 thread)
template <int BS>
__device__ void w_mma(const GemmParams& p, WSmem& sm, uint32_t tmem_base) {
  int stage = 0, us = 0, acc = 0;
  uint32_t phase = 0, uphase = 0, aphase = 0;
  bool ok = true;
  const uint32_t idesc_bf16 = idesc_make(1, W::TM, W::TN);
  const uint32_t idesc_fp8 = idesc_make(0, W::TM, W::TN);
  // B (weights, 256 rows) at the stage base, A (tokens) after the two weight tiles
  const uint64_t desc_b0 = sdesc_sw128(smem_u32(sm.stages));
  const uint64_t desc_a0 = desc_b0 + ((2 * W::W_TILE) >> 4);
  const uint64_t STAGE_D = static_cast<uint64_t>(p.w_stage_bytes) >> 4;
  // accumulator slots: one in block-scaled launches (the scale ring takes the other half of
  // TMEM)
  constexpr int nacc = BS != BS_NONE ? 1 : W::NACC;
  constexpr uint32_t idesc_fp4 = idesc_nv4(W::TM, W::TN);
  while (ok) {
    if (!mbar_wait(&sm.ufull[us], uphase, sm.abort_flag, p.err, p.timeout)) break;
    const WUnit info = sm.ring[us];
    mbar_arrive(&sm.uempty[us]);
    if (++us == W::US) { us = 0; uphase ^= 1; }
    if (info.task < 0) break;
    const GemmTask& T = p.task[info.task];
    if (T.kind == TASK_NORM) continue;  // no tensor-core work
    const int kpg = T.kpg;
    const bool promote = kpg > 0;
    const bool fp8 = T.fp8 != 0;
    const uint32_t idesc = fp8 ? idesc_fp8 : idesc_bf16;
    // (block-scaled launches run routed units only, which are never split in K)
    const int kb0 = BS != BS_NONE ? 0 : info.kb0;
    const int kb1 = BS != BS_NONE ? T.kb_total : info.kb1;
    const bool dual = info.dual != 0;  // two token tiles share the weight operand
    // the slot after `acc` (the second tile of a dual unit) and its phase parity
    const int acc2 = acc + 1 == nacc ? 0 : acc + 1;
    const uint32_t aphase2 = acc + 1 == nacc ? aphase ^ 1 : aphase;
    const bool mxu = BS == BS_MX8 && T.a_sf != nullptr;  // block-scaled FP8 unit
    const bool nvu = BS == BS_NV4 && T.a_sf != nullptr;  // block-scaled FP4 unit
    if (!promote) {
      if (!mbar_wait_spin(&sm.tempty[acc], aphase ^ 1, sm.abort_flag, p.err, p.timeout)) break;
      if (dual &&
          !mbar_wait_spin(&sm.tempty[acc2], aphase2 ^ 1, sm.abort_flag, p.err, p.timeout))
        break;
      tc_fence_after();
    }
    int gpos = 0;  // position of the next k-block in its promotion group
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!mbar_wait_spin(&sm.full[stage], phase, sm.abort_flag, p.err, p.timeout)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (promote && gpos == 0) {
        if (!mbar_wait_spin(&sm.tempty[acc], aphase ^ 1, sm.abort_flag, p.err, p.timeout)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      const uint32_t d = tmem_base + static_cast<uint32_t>(acc * W::TN);
      const uint64_t off = static_cast<uint64_t>(stage) * STAGE_D;
      const uint32_t accum = promote ? static_cast<uint32_t>(gpos > 0)
                                     : static_cast<uint32_t>(kb > kb0);
      if (nvu) {  // (block-scaled units are routed: never split in K, kb0 = 0)
        // this stage's twelve scale tiles into its 48 TMEM columns beside the accumulator:
        // MMA j (K = 64) reads the tokens' at +4j (lane m, column m/32) and the weights'
        // at +16 + 8j (lane n%32, column n/32 over both row blocks), then the four MMAs
        const uint32_t sfc = tmem_base + W::TN + static_cast<uint32_t>(stage * W::NV4_SF_COLS);
        const uint32_t sfs =
            smem_u32(sm.stages + static_cast<size_t>(stage) * p.w_stage_bytes + 2 * W::W_TILE +
                     W::T_TILE);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          tmem_cp_32x128b_x4(sfc + 4 * j, sfs + 512 * j);
          tmem_cp_32x128b_x4(sfc + 16 + 8 * j, sfs + 2048 + 512 * j);
          tmem_cp_32x128b_x4(sfc + 20 + 8 * j, sfs + 4096 + 512 * j);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
          mma_nv4(d, desc_a0 + off + 2 * j, desc_b0 + off + 2 * j, idesc_fp4, sfc + 4 * j,
                  sfc + 16 + 8 * j, static_cast<uint32_t>(kb > 0 || j > 0));
      } else if (mxu) {
        // this stage's scale tiles into its TMEM columns beside the accumulator (tokens:
        // lane m column m/32; weights: lane n%32 column 4 + n/32), then the four K = 32
        // MMAs of the k-block, each with the scale byte of its 32-wide chunk
        const uint32_t sfc = tmem_base + W::TN + static_cast<uint32_t>(stage * W::SF_COLS);
        const uint32_t sfs = smem_u32(sm.sf + stage * W::SF_STAGE);
        tmem_cp_32x128b_x4(sfc, sfs);
        tmem_cp_32x128b_x4(sfc + 4, sfs + 512);
        tmem_cp_32x128b_x4(sfc + 8, sfs + 1024);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          mma_mx(d, desc_a0 + off + 2 * j, desc_b0 + off + 2 * j,
                 idesc_mx(W::TM, W::TN, j, j), sfc, sfc + 4,
                 static_cast<uint32_t>(kb > 0 || j > 0));
      } else if (fp8) {
        mma4_fp8(d, desc_a0 + off, desc_b0 + off, idesc, accum);
      } else {
        mma4_bf16(d, desc_a0 + off, desc_b0 + off, idesc, accum);
      }
      if (dual) {  // second token tile, same weights, into the next slot
        const uint32_t d2 = tmem_base + static_cast<uint32_t>(acc2 * W::TN);
        const uint64_t da2 = desc_a0 + off + (W::T_TILE >> 4);
        if (fp8) mma4_fp8(d2, da2, desc_b0 + off, idesc, accum);
        else mma4_bf16(d2, da2, desc_b0 + off, idesc, accum);
      }
      tc_commit(&sm.empty[stage]);
      if (++stage == p.w_stages) { stage = 0; phase ^= 1; }
      if (promote && ++gpos == kpg) {
        gpos = 0;
        tc_commit(&sm.tfull[acc]);
        if (++acc == nacc) { acc = 0; aphase ^= 1; }
      }
    }
    if (!ok) break;
    if (!promote) {
      tc_commit(&sm.tfull[acc]);
      if (++acc == nacc) { acc = 0; aphase ^= 1; }
      if (dual) {
        tc_commit(&sm.tfull[acc]);
        if (++acc == nacc) { acc = 0; aphase ^= 1; }
      }
    }
  }
  // Drain: all MMAs issued by this thread complete before TMEM is released.
  int dummy_abort = 0;
  tc_commit(sm.drain);
  mbar_wait(sm.drain, 0, &dummy_abort, p.err, p.timeout);
}

// ------------------------------------------------------------------ epilogue
// Unit completion: every epilogue warp arrives (release, CTA scope) on the next slot of
// the signal ring once its writes of the unit are issued; the signalling warp acquires the
// completed phase and publishes with one gpu-scope release add (cumulative over what it
// acquired), so the epilogue never waits for its own writes to become visible.
struct SigState {
  int slot = 0;
  uint32_t phase = 0;
};
__device__ __forceinline__ void w_signal(const GemmParams& p, WSmem& sm, SigState& sg,
                                         int* counter, int ew, int lane) {
  if (lane == 0)  // the slot's previous request has been published
    mbar_wait(&sm.sempty[sg.slot], sg.phase ^ 1, sm.abort_flag, p.err, p.timeout);
  __syncwarp();
  if (ew == 0 && lane == 0) sm.sptr[sg.slot] = counter;
  if (lane == 0) mbar_arrive(&sm.sfull[sg.slot]);
  if (++sg.slot == W::SIG) { sg.slot = 0; sg.phase ^= 1; }
}

__device__ void w_signaller(const GemmParams& p, WSmem& sm) {
  int slot = 0;
  uint32_t phase = 0;
  for (;;) {
    if (!mbar_wait(&sm.sfull[slot], phase, sm.abort_flag, p.err, p.timeout)) return;
    int* counter = sm.sptr[slot];
    if (counter == nullptr) return;  // end of work
    red_release_gpu_add(counter, 1);
    mbar_arrive(&sm.sempty[slot]);
    if (++slot == W::SIG) { slot = 0; phase ^= 1; }
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// One k-split of an output tile (token tile of `rows` tokens x 256 features): this thread's
// 128 fp32 sums (token (ew % 4) * 32 + lane, features [128 half, 128 half + 128) of the tile)
// are added into the tile's fp32 rows of out_acc, 16 features of the warp's 32 tokens at a
// time through the per-warp transpose (8 tokens x 64 contiguous bytes per vector
// reduction).  After a fence, the tile's arrival counter tells the last split, whose
// epilogue warps round the tile to bf16 into out (row by row, coalesced), zero its rows of
// out_acc and its counter for the next forward.
__device__ __forceinline__ void w_out_split(const GemmParams& p, WSmem& sm, const GemmTask& T,
                                         const WUnit& info, int row0, int rows,
                                         const float* a, int ew, int lane) {
  const int half = ew / 4;
  float* st = sm.stg + ew * 32 * STG_LD;
  const int qd = lane & 3;
  // lane: quad qd of warp-local tokens lane / 4 + 8 it (tile rows (ew % 4) * 32 + those)
  float* base = p.out_acc + static_cast<size_t>(row0 + (ew & 3) * 32 + (lane >> 2)) * p.H +
                static_cast<size_t>(info.ftile) * 256 + half * 128 + 4 * qd;
  const int tk0 = (ew & 3) * 32 + (lane >> 2);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<float4*>(st + stg_quad(lane, j)) =
          make_float4(a[16 * c + 4 * j], a[16 * c + 4 * j + 1], a[16 * c + 4 * j + 2],
                      a[16 * c + 4 * j + 3]);
    __syncwarp();
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const float4 v =
          *reinterpret_cast<const float4*>(st + stg_quad(it * 8 + (lane >> 2), qd));
      if (tk0 + 8 * it < rows)
        red_add_v4(base + static_cast<size_t>(8 * it) * p.H + 16 * c, v.x, v.y, v.z, v.w);
    }
    __syncwarp();
  }
  __threadfence();  // this thread's additions before the arrival below
  named_bar_sync(2, W::EPI_THREADS);
  if (ew == 0 && lane == 0) {
    const int tile = info.dep_idx * T.ftiles + info.ftile;
    const int last = atomicAdd(p.out_cnt + tile, 1) == T.ksplit - 1;
    if (last) p.out_cnt[tile] = 0;  // every split has arrived: ready for the next forward
    *reinterpret_cast<volatile int*>(sm.split_last) = last;
  }
  named_bar_sync(2, W::EPI_THREADS);
  if (!*reinterpret_cast<volatile int*>(sm.split_last)) return;
  __threadfence();  // the other splits' additions before the reads below
  // warp ew: tile rows ew, ew + 8, ...; lane: features [8 lane, 8 lane + 8)
  for (int r = ew; r < rows; r += W::EPI_WARPS) {
    float4* acc = reinterpret_cast<float4*>(p.out_acc + static_cast<size_t>(row0 + r) * p.H +
                                            static_cast<size_t>(info.ftile) * 256) +
                  2 * lane;
    const float4 v0 = __ldcg(acc), v1 = __ldcg(acc + 1);
    __stcg(acc, make_float4(0.f, 0.f, 0.f, 0.f));
    __stcg(acc + 1, make_float4(0.f, 0.f, 0.f, 0.f));
    *reinterpret_cast<uint4*>(p.out + static_cast<size_t>(row0 + r) * p.H +
                              static_cast<size_t>(info.ftile) * 256 + 8 * lane) =
        make_uint4(pack_bf16x2(v0.x, v0.y), pack_bf16x2(v0.z, v0.w), pack_bf16x2(v1.x, v1.y),
                   pack_bf16x2(v1.z, v1.w));
  }
}

// RMSNorm of up to NORM_ROWS token rows of the fp32 combine, one row per epilogue warp:
// fp32 statistic (lane partials, then a shuffle tree), gamma applied, one bf16 rounding (the
// output GEMM's token operand).  No barrier between the warps.
template <bool DET>
__device__ void w_norm_rows(const GemmParams& p, WSmem& sm, SigState& sg, int row0, int rows,
                            int ew, int lane) {
  if (ew < rows) {
    const size_t t = static_cast<size_t>(row0 + ew);
    const float4* rv = reinterpret_cast<const float4*>(p.r + t * p.L);
    // the combined row: r (added into by the routed L2 units), or the token's topk weighted
    // slots summed in choice order (deterministic combine)
    auto row4 = [&](int c) {
      if constexpr (!DET) {
        return __ldcg(rv + c);
      } else {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < p.topk; ++j) {
          const int pj = __ldg(p.pos + t * p.topk + j);
          const float4 y =
              __ldcg(reinterpret_cast<const float4*>(p.yw + static_cast<size_t>(pj) * p.L) + c);
          acc.x += y.x;
          acc.y += y.y;
          acc.z += y.z;
          acc.w += y.w;
        }
        return acc;
      }
    };
    const int n4 = p.L / 4;
    constexpr int PER = 32;  // float4s per lane held in registers (L <= 4096)
    float4 v[PER];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int c = lane + i * 32;
      v[i] = c < n4 ? row4(c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < PER; ++i)
      ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
    if constexpr (!DET) {
      // the row is in registers: zero it for the next forward's combine
      if (p.zero_r) {
        float4* rw = reinterpret_cast<float4*>(p.r + t * p.L);
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          const int c = lane + i * 32;
          if (c < n4) rw[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    const float inv = rsqrtf(ss / static_cast<float>(p.L) + p.eps);
    const uint2* gg = reinterpret_cast<const uint2*>(p.gamma);
    uint2* nn = reinterpret_cast<uint2*>(p.nrm + t * p.L);
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int c = lane + i * 32;
      if (c < n4) {
        const float4 x = v[i];
        const uint2 graw = __ldg(gg + c);
        const __nv_bfloat162 g01 = *reinterpret_cast<const __nv_bfloat162*>(&graw.x);
        const __nv_bfloat162 g23 = *reinterpret_cast<const __nv_bfloat162*>(&graw.y);
        const __nv_bfloat162 o01 = __floats2bfloat162_rn(x.x * inv * __low2float(g01),
                                                         x.y * inv * __high2float(g01));
        const __nv_bfloat162 o23 = __floats2bfloat162_rn(x.z * inv * __low2float(g23),
                                                         x.w * inv * __high2float(g23));
        uint2 o;
        o.x = *reinterpret_cast<const uint32_t*>(&o01);
        o.y = *reinterpret_cast<const uint32_t*>(&o23);
        nn[c] = o;
      }
    }
  }
  w_signal(p, sm, sg, p.norm_done + row0 / W::TM, ew, lane);
}

template <bool DET, int BS>
__device__ void w_epilogue(const GemmParams& p, WSmem& sm, uint32_t tmem_base) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ew = warp - W::FIRST_EPI_WARP;
  const int quad = warp & 3;  // TMEM lane quadrant this warp may access
  const int half = ew >> 2;   // column half of this warp
  const int tok = quad * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
  int us = 0, acc = 0, steps = 0, l1_units = 0;
  uint32_t uphase = 0, aphase = 0;
  SigState sg;
  const int G_L = p.L / 128, G_I = p.I / 128;
  constexpr int nacc = BS != BS_NONE ? 1 : W::NACC;

  for (;;) {
    if (!mbar_wait(&sm.ufull[us], uphase, sm.abort_flag, p.err, p.timeout)) return;
    const WUnit info = sm.ring[us];
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.uempty[us]);
    if (++us == W::US) { us = 0; uphase ^= 1; }
    if (info.task < 0) {
      w_signal(p, sm, sg, nullptr, ew, lane);  // releases the signalling warp
      return;
    }
    const GemmTask& T = p.task[info.task];
    const int kind = T.kind;
    if (kind == TASK_NORM) {
      w_norm_rows<DET>(p, sm, sg, info.row0, info.rows, ew, lane);
      continue;
    }
    // a dual unit (two token tiles sharing the weight operand, accumulated in consecutive
    // slots) is finished as two single-tile units
    const int nsub = info.dual ? 2 : 1;
    for (int si = 0; si < nsub; ++si) {
      const int row0 = info.row0 + si * W::TM;
      const int rows = si ? min(W::TM, p.M - row0) : info.rows;
      const int dep_idx = info.dep_idx + si;
      const bool pair = is_pair(kind);
      const bool valid = tok < rows;
      // combine target of a routed L2 row, fetched while the products are computed
      int tg = 0;
      float wv = 0.f;
      if (kind == TASK_ROUTED_L2 && valid) {
        tg = __ldg(p.gidx + row0 + tok);
        wv = __ldg(p.wperm + row0 + tok);
      }
      // TMEM columns of this thread's two 64-column groups
      const uint32_t col0 = pair ? half * 64 : half * 128;
      const uint32_t col1 = pair ? 128 + half * 64 : half * 128 + 64;
      float a[128];

      if (T.kpg > 0) {
        // Block-scaled products: every promotion group's partial (fresh in TMEM) is added
        // with scale = token scale x weight block scale of the group.
  #pragma unroll
        for (int i = 0; i < 128; ++i) a[i] = 0.f;
        const int ng = T.kb_total / T.kpg;
        const float* ts =
            (kind == TASK_ROUTED_L1 ? p.zsT : p.asT) + row0 + tok;
        const float *sw0, *sw1;
        if (kind == TASK_ROUTED_L1) {
          const size_t rb = static_cast<size_t>(info.e) * (2 * G_I);
          sw0 = p.w13_s + (rb + info.ftile) * G_L;
          sw1 = p.w13_s + (rb + G_I + info.ftile) * G_L;
        } else {
          sw0 = p.w2_s + (static_cast<size_t>(info.e) * G_L + 2 * info.ftile + half) * G_I;
          sw1 = sw0;
        }
        // scales are loaded two groups ahead so no global load sits between the
        // accumulator hand-offs
        auto tok_scale = [&](int gi) {
          return valid && gi < ng ? __ldcg(ts + static_cast<size_t>(gi) * p.cap) : 0.f;
        };
        auto w_scale = [&](const float* sw, int gi) { return gi < ng ? __ldg(sw + gi) : 0.f; };
        float sa1 = tok_scale(0), w01 = w_scale(sw0, 0), w11 = w_scale(sw1, 0);
        float sa2 = tok_scale(1), w02 = w_scale(sw0, 1), w12 = w_scale(sw1, 1);
        for (int gi = 0; gi < ng; ++gi) {
          const float s0 = w01 * sa1;
          const float s1 = w11 * sa1;
          sa1 = sa2;
          w01 = w02;
          w11 = w12;
          sa2 = tok_scale(gi + 2);
          w02 = w_scale(sw0, gi + 2);
          w12 = w_scale(sw1, gi + 2);
          if (!mbar_wait_spin(&sm.tfull[acc], aphase, sm.abort_flag, p.err, p.timeout)) return;
          tc_fence_after();
          const uint32_t tb = tmem_base + lane_base + static_cast<uint32_t>(acc * W::TN);
          float v[4][16];
          tmem_ld16x4(tb + col0, tb + col0 + 16, tb + col0 + 32, tb + col0 + 48, v[0], v[1],
                      v[2], v[3]);
  #pragma unroll
          for (int c = 0; c < 4; ++c)
  #pragma unroll
            for (int i = 0; i < 16; ++i) a[c * 16 + i] = fmaf(v[c][i], s0, a[c * 16 + i]);
          tmem_ld16x4(tb + col1, tb + col1 + 16, tb + col1 + 32, tb + col1 + 48, v[0], v[1],
                      v[2], v[3]);
          // the slot's contents are in registers: hand it back before the last FMAs
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.tempty[acc]);
          if (++acc == nacc) { acc = 0; aphase ^= 1; }
  #pragma unroll
          for (int c = 0; c < 4; ++c)
  #pragma unroll
            for (int i = 0; i < 16; ++i)
              a[64 + c * 16 + i] = fmaf(v[c][i], s1, a[64 + c * 16 + i]);
          if (ew == 0 && lane == 0) trace_mark(p, 2, steps++);
        }
      } else {
        if (!mbar_wait_spin(&sm.tfull[acc], aphase, sm.abort_flag, p.err, p.timeout)) return;
        tc_fence_after();
        const uint32_t tb = tmem_base + lane_base + static_cast<uint32_t>(acc * W::TN);
        tmem_ld16x4(tb + col0, tb + col0 + 16, tb + col0 + 32, tb + col0 + 48, a, a + 16,
                    a + 32, a + 48);
        tmem_ld16x4(tb + col1, tb + col1 + 16, tb + col1 + 32, tb + col1 + 48, a + 64, a + 80,
                    a + 96, a + 112);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.tempty[acc]);
        if (++acc == nacc) { acc = 0; aphase ^= 1; }
        if (ew == 0 && lane == 0) trace_mark(p, 2, steps++);
      }

      // ---- unit end (this thread: one token, 64 gate/up pairs or 128 features)
      // NVFP4 units: the weights' fp32 per-matrix scale of this expert (the tensor core
      // applied the per-16 scales); for the routed L2 it folds into the routing weight
      if (BS == BS_NV4 && T.a_g != nullptr && kind == TASK_ROUTED_L2) wv *= __ldg(T.a_g + info.e);
      if (BS == BS_NV4 && kind == TASK_ROUTED_L1) {
        // scale by the expert's fp32 matrix scale, SwiGLU, then NVFP4: per 16 outputs an
        // e4m3 scale s = e4m3(amax / 6) and e2m1 codes of a / s (a zero scale gives zero
        // codes).  This thread's 64 outputs are one 64-wide MMA step of the routed L2, so
        // its four scale bytes are one word of that step's token scale tile.
        const float gw = __ldg(T.a_g + info.e);
  #pragma unroll
        for (int i = 0; i < 64; ++i) a[i] = silu_fast(gw * a[i]) * (gw * a[64 + i]);
        uint32_t sfw = 0x38383838u;  // rows past the tile's pairs: scale 1
        if (valid) {
          uint32_t w8[8];  // 64 codes, two per byte
          sfw = 0;
  #pragma unroll
          for (int b = 0; b < 4; ++b) {
            float m = 0.f;
  #pragma unroll
            for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(a[16 * b + i]));
            const uint32_t sc = f32_to_e4m3(quot_rn(m, 6.0f, 1.0f / 6.0f));
            const float s = e4m3_to_f32(static_cast<uint8_t>(sc));
            const float inv = s != 0.f ? rcp_nr(s) : 0.f;
  #pragma unroll
            for (int q = 0; q < 2; ++q) {
              const float* x = a + 16 * b + 8 * q;
              w8[2 * b + q] =
                  s != 0.f ? f32x8_to_e2m1x8(quot_rn(x[0], s, inv), quot_rn(x[1], s, inv),
                                             quot_rn(x[2], s, inv), quot_rn(x[3], s, inv),
                                             quot_rn(x[4], s, inv), quot_rn(x[5], s, inv),
                                             quot_rn(x[6], s, inv), quot_rn(x[7], s, inv))
                           : 0u;
            }
            sfw |= sc << (8 * b);
          }
          const size_t pp = static_cast<size_t>(row0 + tok);
          uint4* dq = reinterpret_cast<uint4*>(p.aq + pp * (p.I / 2) +
                                               (static_cast<size_t>(info.ftile) * 128 + half * 64) / 2);
          dq[0] = make_uint4(w8[0], w8[1], w8[2], w8[3]);
          dq[1] = make_uint4(w8[4], w8[5], w8[6], w8[7]);
        }
        *reinterpret_cast<uint32_t*>(p.asf_t +
                                     (static_cast<size_t>(dep_idx) * (p.I / 64) +
                                      2 * info.ftile + half) * 512 +
                                     (tok & 31) * 16 + 4 * (tok >> 5)) = sfw;
        if (p.l1_done != nullptr) w_signal(p, sm, sg, p.l1_done + dep_idx, ew, lane);
      } else if (BS == BS_MX8 && kind == TASK_ROUTED_L1) {
        // SwiGLU, then MX e4m3: one power-of-two scale per 32 outputs, 2^(floor(log2 amax)
        // - 8); this thread's 64 outputs are two whole groups, so no other thread is
        // involved.  The scale bytes go to the routed L2 units' token scale tile of this
        // routed tile: k-block = this 128-output tile, chunk = 2 * half + group.
  #pragma unroll
        for (int i = 0; i < 64; ++i) a[i] = silu_fast(a[i]) * a[64 + i];
        int ex[2];
        float inv[2];
  #pragma unroll
        for (int gq = 0; gq < 2; ++gq) {
          float m = 0.f;
  #pragma unroll
          for (int i = 0; i < 32; ++i) m = fmaxf(m, fabsf(a[32 * gq + i]));
          ex[gq] = mx_exponent(m);
          inv[gq] = pow2_exact(-ex[gq]);
        }
        uint32_t sfw = 0x7F7Fu;  // rows past the tile's pairs: scale 1
        if (valid) {
          const size_t pp = static_cast<size_t>(row0 + tok);
          const size_t col = static_cast<size_t>(info.ftile) * 128 + half * 64;
          uint4* dq = reinterpret_cast<uint4*>(p.aq + pp * p.I + col);
  #pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float iv = inv[c >> 1];  // 16 outputs per c: groups of 32 are c = 0,1 | 2,3
            uint32_t w4[4];
  #pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int i = c * 16 + q * 4;
              w4[q] = f32x2_to_e4m3x2(a[i] * iv, a[i + 1] * iv) |
                      (f32x2_to_e4m3x2(a[i + 2] * iv, a[i + 3] * iv) << 16);
            }
            dq[c] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
          sfw = static_cast<uint32_t>(ex[0] + 127) | (static_cast<uint32_t>(ex[1] + 127) << 8);
        }
        uint8_t* tsf = p.asf_t +
                       (static_cast<size_t>(dep_idx) * G_I + info.ftile) * 512 +
                       (tok & 31) * 16 + 4 * (tok >> 5) + 2 * half;
        *reinterpret_cast<uint16_t*>(tsf) = static_cast<uint16_t>(sfw);
        if (p.l1_done != nullptr) w_signal(p, sm, sg, p.l1_done + dep_idx, ew, lane);
      } else if (kind == TASK_ROUTED_L1) {
        // SwiGLU, then e4m3 with one scale per token per 128 outputs (both halves' amax)
        float m = 0.f;
  #pragma unroll
        for (int i = 0; i < 64; ++i) {
          a[i] = silu_fast(a[i]) * a[64 + i];
          m = fmaxf(m, fabsf(a[i]));
        }
        float* am = sm.amax + (l1_units & 1) * 2 * W::TM;
        ++l1_units;
        am[half * W::TM + tok] = m;
        named_bar_sync(1, W::EPI_THREADS);
        const float amax = fmaxf(am[tok], am[W::TM + tok]);
        const float sc = amax == 0.f ? 1.0f : amax / 448.0f;
        const float inv = 1.0f / sc;
        if (valid) {
          const size_t pp = static_cast<size_t>(row0 + tok);
          const size_t col = static_cast<size_t>(info.ftile) * 128 + half * 64;
          uint4* dq = reinterpret_cast<uint4*>(p.aq + pp * p.I + col);
  #pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t w4[4];
  #pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int i = c * 16 + q * 4;
              w4[q] = f32x2_to_e4m3x2(quot_rn(a[i], sc, inv), quot_rn(a[i + 1], sc, inv)) |
                      (f32x2_to_e4m3x2(quot_rn(a[i + 2], sc, inv), quot_rn(a[i + 3], sc, inv))
                       << 16);
            }
            dq[c] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            if (p.aqb != nullptr) {  // exact bf16 images of the codes
              uint4* db = reinterpret_cast<uint4*>(p.aqb + pp * p.I + col) + 2 * c;
              uint32_t b8[8];
  #pragma unroll
              for (int q = 0; q < 8; ++q) {
                const uint32_t wq = w4[q >> 1] >> ((q & 1) * 16);
                b8[q] = pack_bf16x2(e4m3_to_f32(static_cast<uint8_t>(wq & 0xFFu)),
                                    e4m3_to_f32(static_cast<uint8_t>((wq >> 8) & 0xFFu)));
              }
              db[0] = make_uint4(b8[0], b8[1], b8[2], b8[3]);
              db[1] = make_uint4(b8[4], b8[5], b8[6], b8[7]);
            }
          }
          if (half == 0) p.asT[static_cast<size_t>(info.ftile) * p.cap + pp] = sc;
        }
        if (p.l1_done != nullptr) w_signal(p, sm, sg, p.l1_done + dep_idx, ew, lane);
      } else if (kind == TASK_SHARED_L1) {
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(
              p.a_s + static_cast<size_t>(row0 + tok) * p.Is + info.ftile * 128 + half * 64);
  #pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t w4[4];
  #pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int i = c * 8 + q * 2;
              w4[q] = pack_bf16x2(silu_fast(a[i]) * a[64 + i], silu_fast(a[i + 1]) * a[65 + i]);
            }
            dst[c] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
        if (p.sh_done != nullptr) w_signal(p, sm, sg, p.sh_done + dep_idx, ew, lane);
      } else if (kind == TASK_ROUTED_L2) {
        if constexpr (DET) {
          // this pair's weighted output, summed in choice order by the norm: 128 features
          // of one permuted row per thread, 16-byte stores
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(
                p.yw + static_cast<size_t>(row0 + tok) * p.L + info.ftile * 256 + half * 128);
  #pragma unroll
            for (int c = 0; c < 32; ++c)
              dst[c] = make_float4(wv * a[4 * c], wv * a[4 * c + 1], wv * a[4 * c + 2],
                                   wv * a[4 * c + 3]);
          }
        } else {
        // Weighted scatter-combine into the tokens' fp32 rows of r.  A lane holds one token's
        // 128 features; 16 features of the warp's 32 tokens at a time pass through shared
        // memory, so each vector reduction instruction covers 8 tokens x 64 contiguous bytes
        // (8 L2 requests) instead of 32 tokens x 16 bytes.  Lane l reduces quad l % 4 of
        // tokens l / 4 + 8i (i < 4); their target rows are fetched once per unit.
        float* st = sm.stg + ew * 32 * STG_LD;
        const int qd = lane & 3;
        const size_t col0 = static_cast<size_t>(info.ftile) * 256 + half * 128 + 4 * qd;
        float* dst[4];
        int src[4];
        bool ok[4];
  #pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int t = it * 8 + (lane >> 2);
          const int tgt = __shfl_sync(0xFFFFFFFFu, tg, t);
          ok[it] = __shfl_sync(0xFFFFFFFFu, valid ? 1 : 0, t) != 0;
          dst[it] = p.r + static_cast<size_t>(tgt) * p.L + col0;
          src[it] = stg_quad(t, qd);
        }
  #pragma unroll
        for (int c = 0; c < 8; ++c) {
  #pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<float4*>(st + stg_quad(lane, j)) =
                make_float4(wv * a[16 * c + 4 * j], wv * a[16 * c + 4 * j + 1],
                            wv * a[16 * c + 4 * j + 2], wv * a[16 * c + 4 * j + 3]);
          __syncwarp();
  #pragma unroll
          for (int it = 0; it < 4; ++it) {
            const float4 v = *reinterpret_cast<const float4*>(st + src[it]);
            if (ok[it]) red_add_v4(dst[it] + 16 * c, v.x, v.y, v.z, v.w);
          }
          __syncwarp();
        }
        }
        if (p.l2_done != nullptr) w_signal(p, sm, sg, p.l2_done, ew, lane);
      } else if (!DET && BS == BS_NONE && T.ksplit > 1) {  // TASK_OUT, one k-split of a tile
        w_out_split(p, sm, T, info, row0, rows, a, ew, lane);
      } else {  // TASK_OUT
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(
              p.out + static_cast<size_t>(row0 + tok) * p.H + info.ftile * 256 + half * 128);
  #pragma unroll
          for (int c = 0; c < 16; ++c)
            dst[c] = make_uint4(pack_bf16x2(a[c * 8], a[c * 8 + 1]),
                                pack_bf16x2(a[c * 8 + 2], a[c * 8 + 3]),
                                pack_bf16x2(a[c * 8 + 4], a[c * 8 + 5]),
                                pack_bf16x2(a[c * 8 + 6], a[c * 8 + 7]));
        }
      }
    }
  }
}

template <bool DET, int BS>
__global__ void __launch_bounds__(W::THREADS, 1) wide_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  WSmem sm(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < W::STAGES; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int a = 0; a < W::NACC; ++a) {
      mbar_init(&sm.tfull[a], 1);
      mbar_init(&sm.tempty[a], W::EPI_WARPS);
    }
    for (int u = 0; u < W::US; ++u) {
      mbar_init(&sm.ufull[u], 1);
      mbar_init(&sm.uempty[u], 1 + W::EPI_WARPS);
    }
    for (int g = 0; g < W::SIG; ++g) {
      mbar_init(&sm.sfull[g], W::EPI_WARPS);
      mbar_init(&sm.sempty[g], 1);
    }
    mbar_init(sm.drain, 1);
    *sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int t = 0; t < p.ntasks; ++t) {
      tma_prefetch_desc(&p.task[t].tmB[0]);
      tma_prefetch_desc(&p.task[t].tmB[1]);
    }
  }
  if (warp == 1) {
    tmem_alloc(sm.tmem_holder, W::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_holder;

  // Everything above touches only this CTA's resources, and the L2 prefetch below only
  // handle-owned weights that no kernel writes; inputs written by the previous kernels in
  // the stream are read only after the wait.
  if (warp == 0 && lane == 0) prefetch_share_l2(p);
  pdl_wait();
  pdl_trigger();

  // Routing tile offsets for the producer's unit decode, read once per CTA by warp 0
  // before the control warps give up registers.
  __shared__ int s_tile_off[MAX_E + 1], s_off[MAX_E + 1];
  int u0 = 0;
  if (warp == 0) {
    // the first unit claim and the offset loads are issued together (all independent),
    // so the launch pays one round trip before its first copy instead of several
    u0 = lane == 0 ? atomicAdd(p.sched, 1) : 0;
    constexpr int NL = (MAX_E + 1 + 31) / 32;
    int to[NL], of[NL];
#pragma unroll
    for (int i = 0; i < NL; ++i) {
      const int k = lane + 32 * i;
      to[i] = k <= p.E ? p.tile_off[k] : 0;
      of[i] = k <= p.E ? p.off[k] : 0;
    }
#pragma unroll
    for (int i = 0; i < NL; ++i) {
      const int k = lane + 32 * i;
      if (k <= p.E) {
        s_tile_off[k] = to[i];
        s_off[k] = of[i];
      }
    }
    __syncwarp();
  }
  if (warp < W::FIRST_EPI_WARP) {
    regs_dec<W::REGS_CTRL>();
    if (warp == 0) {
      if (lane == 0) w_producer<BS>(p, sm, s_tile_off, s_off, u0);
    } else if (warp == 1) {
      if (lane == 0) w_mma<BS>(p, sm, tmem_base);
    } else if (warp == W::SIGNAL_WARP) {
      if (lane == 0) w_signaller(p, sm);
    }
  } else {
    regs_inc<W::REGS_EPI>();
    w_epilogue<DET, BS>(p, sm, tmem_base);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, W::TMEM_COLS);
  }
}

}  // namespace

static_assert(WSmem::bytes() + 2 * (MAX_E + 1) * 4 <= 227 * 1024, "shared memory budget");

// The six instantiations: deterministic combine or not x no block scale, MX, NVFP4.
const void* wide_fn(bool det, int bs) {
  if (det)
    return bs == BS_MX8   ? reinterpret_cast<const void*>(wide_kernel<true, BS_MX8>)
           : bs == BS_NV4 ? reinterpret_cast<const void*>(wide_kernel<true, BS_NV4>)
                          : reinterpret_cast<const void*>(wide_kernel<true, BS_NONE>);
  return bs == BS_MX8   ? reinterpret_cast<const void*>(wide_kernel<false, BS_MX8>)
         : bs == BS_NV4 ? reinterpret_cast<const void*>(wide_kernel<false, BS_NV4>)
                        : reinterpret_cast<const void*>(wide_kernel<false, BS_NONE>);
}

int wide_kernel_regs() {  // every instantiation must launch with the planned registers
  const void* k[] = {wide_fn(false, BS_NONE), wide_fn(true, BS_NONE), wide_fn(false, BS_MX8),
                     wide_fn(true, BS_MX8),   wide_fn(false, BS_NV4), wide_fn(true, BS_NV4)};
  int regs = -1;
  for (const void* f : k) {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, f) != cudaSuccess) return -1;
    if (regs >= 0 && a.numRegs != regs) return -1;
    regs = a.numRegs;
  }
  return regs;
}

bool wide_regs_ok(int regs) { return regs == W::LAUNCH_REGS; }

cudaError_t launch_wide(const GemmParams& p, int grid, cudaStream_t s, bool pdl) {
  const int smem = WSmem::bytes();
  // the deterministic combine and the block-scaled launches are instantiations of their own
  const void* f = wide_fn(p.yw != nullptr, p.bs);
  cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(W::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  void* args[] = {const_cast<GemmParams*>(&p)};
  return cudaLaunchKernelExC(&cfg, f, args);
}

}  // namespace klt
