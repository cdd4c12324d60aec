// Persistent tile engine of the latent-MoE tail on sm_103a (tcgen05 + TMEM + TMA).
//
// One kernel serves every GEMM of the tail.  A launch carries up to two tasks; its
// persistent CTAs pull work units (one 128-row output tile x one token tile x one K
// range) from a device counter, so routed expert tiles and shared-expert tiles of one
// launch interleave on the SMs the way the MegaMoE scheduler co-schedules routed and
// shared L1/L2 work (DeepGEMM PR 416, Implementation).
//
// Orientation: the weight matrix is the MMA "A" operand (128 output features per tile,
// one TMEM lane each) and the tokens are the "B" operand (BN columns), so a decode batch
// of a few tokens still fills the 128-row MMA and the kernel streams weights.
//
// Roles per CTA (1 CTA per SM, 12 warps):
//   warp 0      TMA producer: decodes units, publishes them to a ring, streams A/B tiles
//               (128-byte swizzled K-major, 128 bytes of K per stage) into STAGES buffers;
//   warp 1      MMA issuer (one thread): tcgen05.mma into TMEM accumulator slots;
//   warps 2, 3  completion signallers (one per epilogue group);
//   warps 4-11  epilogue: TMEM -> registers, then the task's fused epilogue; up to 32-token
//               tiles two groups of four warps take alternate units.
//
// FP8 routed tasks use per-128-K promotion: every 128-wide K block is accumulated by the
// tensor core into its own TMEM slot and the epilogue adds it into fp32 registers scaled
// by (weight block scale x token group scale), because the scales are general fp32 and
// no hardware block-scaled MMA takes them.  BF16 tasks accumulate the whole K range in
// TMEM.  Every wait is bounded; an expired wait raises the CTA abort flag and the sticky
// device error, and the CTA drains its own copies and MMAs before freeing TMEM.
#include "klt_device.cuh"
#include "klt_internal.h"

namespace klt {

namespace {

template <int BN>
struct Cfg {
  // Warp roles (3 warpgroups): warp 0 = TMA producer, warp 1 = MMA issuer, warps 2 and 3 =
  // completion signallers (one per epilogue group), warps 4..11 = epilogue.  Up to 32-token
  // tiles the eight epilogue warps form two groups of four that take alternate work units,
  // so two units' epilogues (scale staging, promotion, combine, signal) overlap on every
  // SM; wider tiles use one group of eight split by column halves.
  static constexpr int EPI_WARPS = 8;
  static constexpr int FIRST_EPI_WARP = 4;
  static constexpr int NGROUPS = BN <= 32 ? 2 : 1;
  static constexpr int GROUP_WARPS = EPI_WARPS / NGROUPS;
  static constexpr int GROUP_THREADS = GROUP_WARPS * 32;
  static constexpr int SIGNAL_WARP = 2;  // + group index
  static constexpr int THREADS = 12 * 32;
  static constexpr int SIG = 8;  // completion-signal ring per group (epilogue -> signaller)
  static constexpr int EPI_THREADS = EPI_WARPS * 32;
  // Registers: 384 threads launch with 168 each; the control warpgroup (producer, MMA
  // issuer, signallers) drops to 88 and the two epilogue warpgroups rise to 208, within
  // the registers released.
  static constexpr int LAUNCH_REGS = 168;
  static constexpr int REGS_CTRL = 88;
  static constexpr int REGS_EPI = 208;
  static_assert(4 * (LAUNCH_REGS - REGS_CTRL) >= 8 * (REGS_EPI - LAUNCH_REGS),
                "register hand-over must balance");
  static constexpr int A_BYTES = 128 * 128;
  static constexpr int B_BYTES = BN * 128;
  // Single-tile tasks carry two k-blocks per stage (A0/A1 + B0/B1) when the stage fits,
  // so every stage keeps ~32 KB of weights in flight.
  static constexpr bool DUAL = BN <= 32;
  static constexpr int STAGE_BYTES = 2 * A_BYTES + (DUAL ? 2 : 1) * B_BYTES;
  static constexpr int STAGES = BN == 16 ? 6 : (BN == 128 ? 3 : 5);
  static_assert(BN == 16 || BN == 32 || BN == 64 || BN == 128, "tile width");
  static constexpr int SLOT_COLS = 2 * BN;
  static constexpr int TMEM_COLS = 512;  // the whole TMEM: 16 accumulator slots at BN=16
  static constexpr int NACC = TMEM_COLS / SLOT_COLS;
  static constexpr int US = 8;
  static constexpr int COLS = BN / (GROUP_WARPS / 4);
  // per-unit scale staging: token group scales [MAX_KB][BN] + weight scales [MAX_KB][2]
  // plus, for the combine, the token index and routing weight of each column [2][BN]
  static constexpr int SC_FLOATS = MAX_KB * BN + 2 * MAX_KB + 2 * BN;
  static_assert(COLS % 16 == 0, "epilogue works in 16-column chunks");
  static_assert(NACC >= 2, "need two accumulator slots");
};

struct UnitInfo {
  int task;   // -1: no more work
  int e;      // routed expert
  int row0;   // first token row of the B tile
  int rows;   // valid token rows (D columns)
  int ftile;  // 128-row output tile
  int arb;    // 128-row block of the (gate) weight tile
  int kb0, kb1;
  int tile_id;   // split-K / stream-K tile (non-routed)
  int split;     // fixed split index
  int ncontrib;  // units contributing to this tile (1: no partials)
  int cfirst;    // stream-K: first contributing CTA
  int wslot;     // stream-K: this unit's partial slot
  int dep_idx;   // routed token tile (routed tasks) or token tile (others)
};

// Stream-K helpers: CTA c owns k-blocks [b(c), b(c+1)) of the task's flattened
// (tile, kb) sequence, b(c) = c * total / grid.
__device__ __forceinline__ long long sk_begin(long long total, int grid, int c) {
  return static_cast<long long>(c) * total / grid;
}
__device__ __forceinline__ int sk_owner(long long total, int grid, long long x) {
  return static_cast<int>(((x + 1) * grid + total - 1) / total - 1);
}
// Partial slot of CTA c for tile t: 0 for its first tile, 1 for its last.
__device__ __forceinline__ int sk_slot(long long total, int grid, int kb_per_tile, int c,
                                       int t) {
  const int first_tile = static_cast<int>(sk_begin(total, grid, c) / kb_per_tile);
  return c * 2 + (t == first_tile ? 0 : 1);
}

template <int BN>
struct Smem {
  using C = Cfg<BN>;
  uint8_t* stages;
  uint64_t *full, *empty, *tfull, *tempty, *ufull, *uempty, *sfull, *sempty, *drain;
  int** sptr;  // [NGROUPS][SIG] counter each completion signal increments (null: end)
  UnitInfo* ring;
  uint32_t* tmem_holder;
  int* abort_flag;
  int* last_flag;  // [NGROUPS]
  float* red;  // [EPI_WARPS][COLS]
  float* sc;   // [NGROUPS][SC_FLOATS] per-unit scale staging of each group

  static constexpr int NSIG = C::NGROUPS * C::SIG;
  static constexpr int BAR_BYTES =
      8 * (2 * C::STAGES + 2 * C::NACC + 2 * C::US + 2 * NSIG + 1) + 8 * NSIG;
  static constexpr int bytes() {
    return C::STAGES * C::STAGE_BYTES + BAR_BYTES + C::US * (int)sizeof(UnitInfo) + 64 +
           C::EPI_WARPS * C::COLS * 4 + C::NGROUPS * C::SC_FLOATS * 4 +
           1024 /* alignment slack */;
  }
  __device__ explicit Smem(uint8_t* raw) {
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023));
    stages = base;
    uint64_t* b = reinterpret_cast<uint64_t*>(base + C::STAGES * C::STAGE_BYTES);
    full = b;
    empty = full + C::STAGES;
    tfull = empty + C::STAGES;
    tempty = tfull + C::NACC;
    ufull = tempty + C::NACC;
    uempty = ufull + C::US;
    sfull = uempty + C::US;
    sempty = sfull + NSIG;
    drain = sempty + NSIG;
    sptr = reinterpret_cast<int**>(drain + 1);
    ring = reinterpret_cast<UnitInfo*>(sptr + NSIG);
    tmem_holder = reinterpret_cast<uint32_t*>(ring + C::US);
    abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
    last_flag = abort_flag + 1;
    red = reinterpret_cast<float*>(tmem_holder + 16);
    sc = red + C::EPI_WARPS * C::COLS;
  }
};

// Optional event trace: stamp i of role r for this CTA.
__device__ __forceinline__ void trace_mark(const GemmParams& p, int role, int i) {
  if (p.trace != nullptr && i < p.trace_n)
    p.trace[(static_cast<long long>(blockIdx.x) * 4 + role) * p.trace_n + i] = global_ns();
}

template <int BN>
__device__ UnitInfo decode_unit(const GemmParams& p, const int* s_tile_off, const int* s_off,
                                int u) {
  UnitInfo info;
  info.task = -1;
  for (int ti = 0; ti < p.ntasks; ++ti) {
    const GemmTask& T = p.task[ti];
    if (T.routed) {
      const int ntiles = s_tile_off[p.E];
      const int per_t = T.ftiles * T.ksplit;
      const int units = ntiles * per_t;
      if (u < units) {
        const int t = u / per_t;
        const int rem = u - t * per_t;
        const int ft = rem / T.ksplit;
        const int sp = rem - ft * T.ksplit;
        int lo = 0, hi = p.E - 1;  // largest e with tile_off[e] <= t
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (s_tile_off[mid] <= t) lo = mid; else hi = mid - 1;
        }
        const int e = lo;
        info.task = ti;
        info.e = e;
        info.row0 = s_off[e] + (t - s_tile_off[e]) * BN;
        info.rows = min(BN, s_off[e + 1] - info.row0);
        info.ftile = ft;
        info.arb = e * T.a_rb_expert + ft * T.a_rb_step;
        info.kb0 = sp * T.kb_per_split;
        info.kb1 = min(T.kb_total, info.kb0 + T.kb_per_split);
        info.tile_id = T.ws_tile_base + t * T.ftiles + ft;
        info.split = sp;
        info.ncontrib = T.ksplit;
        info.cfirst = 0;
        info.wslot = 0;
        info.dep_idx = t;
        return info;
      }
      u -= units;
    } else {
      if (u < T.units && T.kind == TASK_NORM) {
        info.task = ti;
        info.e = 0;
        info.row0 = u;
        info.rows = 1;
        info.ftile = 0;
        info.arb = 0;
        info.kb0 = info.kb1 = 0;
        info.tile_id = 0;
        info.split = 0;
        info.ncontrib = 1;
        info.cfirst = 0;
        info.wslot = 0;
        info.dep_idx = u / BN;
        return info;
      }
      if (u < T.units) {
        const int per_n = T.ftiles * T.ksplit;
        const int nt = u / per_n;
        const int rem = u - nt * per_n;
        const int ft = rem / T.ksplit;
        const int sp = rem - ft * T.ksplit;
        info.task = ti;
        info.e = 0;
        info.row0 = nt * BN;
        info.rows = min(BN, p.M - info.row0);
        info.ftile = ft;
        info.arb = ft * (T.a_rb_step > 0 ? T.a_rb_step : 1);
        info.kb0 = T.kb_lo + sp * T.kb_per_split;
        info.kb1 = min(T.kb_total, info.kb0 + T.kb_per_split);
        info.tile_id = T.ws_tile_base + nt * T.ftiles + ft;
        // a tile's K range may be shared out between two tasks: contributions are numbered
        // over both, so the last arriver sums every partial in one fixed order
        info.split = T.split_base + sp;
        info.ncontrib = T.ncontrib > 0 ? T.ncontrib : T.ksplit;
        info.cfirst = 0;
        info.wslot = 0;
        info.dep_idx = nt;
        return info;
      }
      u -= T.units;
    }
  }
  return info;
}

// Next stream-K piece of this CTA (task 0); advances the cursor x.
template <int BN>
__device__ UnitInfo next_streamk_piece(const GemmParams& p, long long& x, long long end) {
  UnitInfo info;
  info.task = -1;
  if (x >= end) return info;
  const GemmTask& T = p.task[0];
  const int K = T.kb_total;
  const int t = static_cast<int>(x / K);
  const int kb0 = static_cast<int>(x - static_cast<long long>(t) * K);
  const int kb1 = static_cast<int>(min(static_cast<long long>(K), kb0 + (end - x)));
  x += kb1 - kb0;
  const int nt = t / T.ftiles, ft = t - nt * T.ftiles;
  info.task = 0;
  info.e = 0;
  info.row0 = nt * BN;
  info.rows = min(BN, p.M - info.row0);
  info.ftile = ft;
  info.arb = ft;
  info.kb0 = kb0;
  info.kb1 = kb1;
  info.tile_id = T.ws_tile_base + t;
  info.split = 0;
  info.cfirst = sk_owner(T.sk_total, T.sk_grid, static_cast<long long>(t) * K);
  info.ncontrib =
      sk_owner(T.sk_total, T.sk_grid, static_cast<long long>(t + 1) * K - 1) - info.cfirst + 1;
  info.wslot = sk_slot(T.sk_total, T.sk_grid, K, blockIdx.x, t);
  info.dep_idx = nt;
  return info;
}

// Bounded wait until the unit's inputs produced by other units of this launch are complete.
// The acquire loads pair with the producers' release adds; the proxy fence orders the
// acquired data before this thread's TMA reads of it.
// One look at whether the unit's inputs produced by other units of this launch are
// complete (acquire loads pairing with the producers' release adds).
template <int BN>
__device__ __forceinline__ bool dep_ready(const GemmParams& p, int dep, int idx,
                                          const int* s_tile_off) {
  if (dep == DEP_L1_TILE) return ld_acquire_gpu(p.l1_done + idx) >= p.l1_target;
  if (dep == DEP_ALL_L2) return ld_acquire_gpu(p.l2_done) >= s_tile_off[p.E] * p.l2_ftiles;
  if (dep == DEP_SH_TILE) return ld_acquire_gpu(p.sh_done + idx) >= p.sh_target;
  if (dep == DEP_NORM_TILE)
    return ld_acquire_gpu(p.norm_done + idx) >= min(BN, p.M - idx * BN);
  return ld_acquire_gpu(p.norm_done + idx) >= min(BN, p.M - idx * BN) &&
         ld_acquire_gpu(p.sh_done + idx) >= p.sh_target;
}

// Bounded wait until the unit's inputs produced by other units of this launch are complete.
// The proxy fence orders the acquired data before this thread's TMA reads of it.
template <int BN>
__device__ bool wait_dependency(const GemmParams& p, int dep, int idx, const int* s_tile_off,
                                volatile int* abort_flag) {
  if (dep == DEP_NONE) return true;
  const long long t0 = clock64();
  while (!dep_ready<BN>(p, dep, idx, s_tile_off)) {
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
template <int BN>
__device__ void run_producer(const GemmParams& p, Smem<BN>& sm, const int* s_tile_off,
                             const int* s_off, int u0) {
  using C = Cfg<BN>;
  const uint64_t pol_w = policy_evict_first();
  const uint64_t pol_t = policy_evict_last();
  int stage = 0, us = 0;
  uint32_t phase = 0, uphase = 0;
  long long issued = 0;
  int published = 0;
  int dummy_abort = 0;
  bool stalled = false;
  const bool streamk = p.task[0].streamk != 0;
  long long sk_x = 0, sk_end = 0;
  int u = u0;  // first unit, claimed by the caller
  if (streamk) {
    if (static_cast<int>(blockIdx.x) < p.task[0].sk_grid) {
      sk_x = sk_begin(p.task[0].sk_total, p.task[0].sk_grid, blockIdx.x);
      sk_end = sk_begin(p.task[0].sk_total, p.task[0].sk_grid, blockIdx.x + 1);
    }
  }
  for (;;) {
    UnitInfo info;
    if (streamk) {
      info = next_streamk_piece<BN>(p, sk_x, sk_end);
    } else {
      info = decode_unit<BN>(p, s_tile_off, s_off, u);
      // claim the next unit now so the counter round trip overlaps this unit's copies
      if (info.task >= 0) u = atomicAdd(p.sched, 1);
    }
    if (info.task < 0) {
      if (mbar_wait(&sm.uempty[us], uphase ^ 1, sm.abort_flag, p.err, p.timeout)) {
        sm.ring[us] = info;
        mbar_arrive(&sm.ufull[us]);
      }
      break;
    }
    const GemmTask& T = p.task[info.task];
    const bool pair = T.pair != 0;
    const int elems_per_kb = T.fp8 ? 128 : 64;
    const int step = (pair || !C::DUAL) ? 1 : 2;
    auto stage_bytes = [&](int nsub) -> uint32_t {
      return pair ? 2 * C::A_BYTES + C::B_BYTES
                  : static_cast<uint32_t>(nsub) * (C::A_BYTES + C::B_BYTES);
    };
    auto issue_a = [&](int kb, int nsub, uint8_t* st, uint64_t* bar) {
      for (int sub = 0; sub < nsub; ++sub) {
        const int kbs = kb + sub;
        const int m = kbs < T.kb_split0 ? 0 : 1;
        const int kk = m ? kbs - T.kb_split0 : kbs;
        // weights are stored pre-swizzled tile-major: one contiguous 16 KB image per
        // (row block, kb), copied as is
        bulk_load(st + sub * C::A_BYTES,
                  T.a_ptr[m] + (static_cast<size_t>(info.arb) * T.a_kb[m] + kk) * C::A_BYTES,
                  C::A_BYTES, bar, pol_w);
        if (pair)
          bulk_load(st + C::A_BYTES,
                    T.a_ptr[m] + (static_cast<size_t>(info.arb + T.a_rb_up) * T.a_kb[m] + kk) *
                                     C::A_BYTES,
                    C::A_BYTES, bar, pol_w);
      }
    };
    auto issue_b = [&](int kb, int nsub, uint8_t* st, uint64_t* bar) {
      for (int sub = 0; sub < nsub; ++sub) {
        const int kbs = kb + sub;
        const int m = kbs < T.kb_split0 ? 0 : 1;
        const int kk = m ? kbs - T.kb_split0 : kbs;
        tma_load_2d(st + 2 * C::A_BYTES + sub * C::B_BYTES, &T.tmB[m], bar, kk * elems_per_kb,
                    info.row0, pol_t);
      }
    };
    int kb = info.kb0;
    if (T.dep != DEP_NONE && dep_ready<BN>(p, T.dep, info.dep_idx, s_tile_off)) {
      // inputs already complete: publish at once, stream weight and token tiles together
      fence_proxy_async_global();
    } else if (T.dep != DEP_NONE) {
      // Stream the unit's weight tiles into the stages that are free now, then wait for
      // the token operand's producers, then copy the token tiles of those stages.
      // the early stages are consecutive ring slots from st0 holding k-blocks kb0, kb0 +
      // step, ...
      const int st0 = stage;
      int npre = 0;
      while (kb < info.kb1 && npre < C::STAGES) {
        if (p.stall_after > 0 && issued >= p.stall_after) break;
        if (!mbar_try_wait(&sm.empty[stage], phase ^ 1)) break;
        const int nsub = min(step, info.kb1 - kb);
        uint8_t* st = sm.stages + stage * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&sm.full[stage], stage_bytes(nsub));
        issue_a(kb, nsub, st, &sm.full[stage]);
        ++npre;
        trace_mark(p, 0, static_cast<int>(issued));
        ++issued;
        if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        kb += step;
      }
      if (!wait_dependency<BN>(p, T.dep, info.dep_idx, s_tile_off, sm.abort_flag)) break;
      for (int i = 0, s = st0, k = info.kb0; i < npre; ++i, k += step) {
        issue_b(k, min(step, info.kb1 - k), sm.stages + s * C::STAGE_BYTES, &sm.full[s]);
        if (++s == C::STAGES) s = 0;
      }
    }
    if (!mbar_wait(&sm.uempty[us], uphase ^ 1, sm.abort_flag, p.err, p.timeout)) break;
    sm.ring[us] = info;
    mbar_arrive(&sm.ufull[us]);
    if (++us == C::US) { us = 0; uphase ^= 1; }
    if (p.trace != nullptr && published < p.trace_n) {  // unit publish time and task
      p.trace[(static_cast<long long>(blockIdx.x) * 4 + 1) * p.trace_n + published] = global_ns();
      p.trace[(static_cast<long long>(blockIdx.x) * 4 + 3) * p.trace_n + published] =
          info.task + 1;
    }
    ++published;
    for (; kb < info.kb1; kb += step) {
      if (p.stall_after > 0 && issued >= p.stall_after) { stalled = true; break; }
      if (!mbar_wait(&sm.empty[stage], phase ^ 1, sm.abort_flag, p.err, p.timeout)) {
        stalled = true;
        break;
      }
      const int nsub = min(step, info.kb1 - kb);
      uint8_t* st = sm.stages + stage * C::STAGE_BYTES;
      mbar_arrive_expect_tx(&sm.full[stage], stage_bytes(nsub));
      issue_a(kb, nsub, st, &sm.full[stage]);
      issue_b(kb, nsub, st, &sm.full[stage]);
      trace_mark(p, 0, static_cast<int>(issued));
      ++issued;
      if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
    }
    if (stalled) break;
  }
  // Drain: wait (bounded, ignoring the abort flag) for this thread's last copies, so no
  // TMA write into shared memory outlives the CTA.
  const long long first = issued > C::STAGES ? issued - C::STAGES : 0;
  for (long long i = first; i < issued; ++i) {
    const int s = static_cast<int>(i % C::STAGES);
    const uint32_t par = static_cast<uint32_t>((i / C::STAGES) & 1);
    mbar_wait(&sm.full[s], par, &dummy_abort, p.err, p.timeout);
  }
}

// ------------------------------------------------------------------ MMA issuer (1 thread)
// The issuing thread pays for every instruction it executes between MMAs, so the loop keeps
// only barrier waits, descriptor adds and the MMAs themselves: per-stage descriptors are
// precomputed, task fields are read once per unit and group positions are counted.
template <int BN>
__device__ void run_mma(const GemmParams& p, Smem<BN>& sm, uint32_t tmem_base) {
  using C = Cfg<BN>;
  int stage = 0, us = 0, acc = 0;
  uint32_t phase = 0, uphase = 0, aphase = 0;
  bool ok = true;
  const uint32_t idesc_bf16 = idesc_make(1, 128, BN);
  const uint32_t idesc_fp8 = idesc_make(0, 128, BN);
  // descriptor of stage 0's A0 tile; every other operand is a fixed offset from it
  const uint64_t desc0 = sdesc_sw128(smem_u32(sm.stages));
  constexpr uint64_t STAGE_D = C::STAGE_BYTES >> 4;
  constexpr uint64_t A_D = C::A_BYTES >> 4;
  constexpr uint64_t B_D = C::B_BYTES >> 4;
  while (ok) {
    if (!mbar_wait(&sm.ufull[us], uphase, sm.abort_flag, p.err, p.timeout)) break;
    const UnitInfo info = sm.ring[us];
    mbar_arrive(&sm.uempty[us]);
    if (++us == C::US) { us = 0; uphase ^= 1; }
    if (info.task < 0) break;
    const GemmTask& T = p.task[info.task];
    if (T.kind == TASK_NORM) continue;  // no tensor-core work
    const bool pair = T.pair != 0;
    const int kpg = T.kpg;
    const bool promote = kpg > 0;
    const bool fp8 = T.fp8 != 0;
    const uint32_t idesc = fp8 ? idesc_fp8 : idesc_bf16;
    const int step = (pair || !C::DUAL) ? 1 : 2;
    const int kb0 = info.kb0, kb1 = info.kb1;
    if (!promote) {
      if (!mbar_wait(&sm.tempty[acc], aphase ^ 1, sm.abort_flag, p.err, p.timeout)) break;
      tc_fence_after();
    }
    int gpos = 0;  // position of the next k-block in its promotion group
    for (int kb = kb0; kb < kb1 && ok; kb += step) {
      if (!mbar_wait(&sm.full[stage], phase, sm.abort_flag, p.err, p.timeout)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int nsub = min(step, kb1 - kb);
      const uint64_t ds = desc0 + static_cast<uint64_t>(stage) * STAGE_D;
      for (int sub = 0; sub < nsub; ++sub) {
        if (promote && gpos == 0) {
          if (!mbar_wait(&sm.tempty[acc], aphase ^ 1, sm.abort_flag, p.err, p.timeout)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * C::SLOT_COLS);
        const uint64_t da = ds + static_cast<uint64_t>(sub) * A_D;
        const uint64_t du = ds + A_D;
        const uint64_t db = ds + 2 * A_D + static_cast<uint64_t>(sub) * B_D;
        const uint32_t accum = promote ? static_cast<uint32_t>(gpos > 0)
                                       : static_cast<uint32_t>(kb + sub > kb0);
        if (fp8) {
          if (pair) mma8_fp8(d, da, du, db, idesc, accum, BN);
          else mma4_fp8(d, da, db, idesc, accum);
        } else {
          if (pair) mma8_bf16(d, da, du, db, idesc, accum, BN);
          else mma4_bf16(d, da, db, idesc, accum);
        }
        if (promote) {
          if (++gpos == kpg) {
            gpos = 0;
            tc_commit(&sm.tfull[acc]);
            if (++acc == C::NACC) { acc = 0; aphase ^= 1; }
          }
        }
      }
      tc_commit(&sm.empty[stage]);
      if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
    }
    if (!ok) break;
    if (!promote) {
      tc_commit(&sm.tfull[acc]);
      if (++acc == C::NACC) { acc = 0; aphase ^= 1; }
    }
  }
  // Drain: all MMAs issued by this thread complete before TMEM is released.
  int dummy_abort = 0;
  tc_commit(sm.drain);
  mbar_wait(sm.drain, 0, &dummy_abort, p.err, p.timeout);
}

// ------------------------------------------------------------------ epilogue
// Unit completion: every epilogue warp arrives (release, CTA scope) on the next slot of the
// signal ring once its writes of the unit are issued; the signalling warp acquires the
// completed phase and publishes with one gpu-scope release add (cumulative over what it
// acquired; the consumer acquires and orders its later TMA reads with a proxy fence), so
// the epilogue never waits for its own writes to become visible.
struct SigState {
  int slot = 0;
  uint32_t phase = 0;
};
// Epilogue group `grp` publishes one unit on its own ring; `gw` is the warp within the group.
template <int BN>
__device__ __forceinline__ void signal_done(const GemmParams& p, Smem<BN>& sm, SigState& sg,
                                            int* counter, int grp, int gw, int lane) {
  using C = Cfg<BN>;
  const int slot = grp * C::SIG + sg.slot;
  if (lane == 0)  // the slot's previous request has been published
    mbar_wait(&sm.sempty[slot], sg.phase ^ 1, sm.abort_flag, p.err, p.timeout);
  __syncwarp();
  if (gw == 0 && lane == 0) sm.sptr[slot] = counter;
  if (lane == 0) mbar_arrive(&sm.sfull[slot]);
  if (++sg.slot == C::SIG) { sg.slot = 0; sg.phase ^= 1; }
}

// Publishes the completions of epilogue group `grp`, in its order, until its end marker.
template <int BN>
__device__ void run_signaller(const GemmParams& p, Smem<BN>& sm, int grp) {
  using C = Cfg<BN>;
  int slot = 0;
  uint32_t phase = 0;
  for (;;) {
    const int s = grp * C::SIG + slot;
    if (!mbar_wait(&sm.sfull[s], phase, sm.abort_flag, p.err, p.timeout)) return;
    int* counter = sm.sptr[s];
    if (counter == nullptr) return;  // end of work
    red_release_gpu_add(counter, 1);
    mbar_arrive(&sm.sempty[s]);
    if (++slot == C::SIG) { slot = 0; phase ^= 1; }
  }
}


// One promotion batch of up to MAXNB groups (fewer when COLS is wide or the unit ends):
// acc += partial * (weight block scale * token group scale), per group.  Returns the
// number of groups consumed, 0 if a bounded wait expired.
template <int BN, int COLS, int MAXNB, bool PAIR>
__device__ __forceinline__ int promote_batch(int left, int kbi, const float* sb, float* g,
                                             float* u, Smem<BN>& sm, uint32_t tmem_base,
                                             uint32_t lane_base, int c0, int& acc,
                                             uint32_t& aphase, const GemmParams& p) {
  using C = Cfg<BN>;
  // registers per thread for one batch: NB groups x (PAIR ? 2 : 1) x 16 columns <= 64
  constexpr int CAP = 64 / ((PAIR ? 2 : 1) * 16);
  constexpr int NBMAX = (COLS == 16) ? (MAXNB < CAP ? MAXNB : CAP) : 1;
  const int nb = left < NBMAX ? left : NBMAX;
  uint32_t tb[4];
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    if (b >= nb) break;
    int slot = acc + b;
    uint32_t par = aphase;
    if (slot >= C::NACC) { slot -= C::NACC; par ^= 1; }
    if (!mbar_wait(&sm.tfull[slot], par, sm.abort_flag, p.err, p.timeout)) return 0;
    tb[b] = tmem_base + lane_base + static_cast<uint32_t>(slot * C::SLOT_COLS);
  }
  tc_fence_after();
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int ch = 0; ch < COLS / 16; ++ch) {
    float v[4][16];
    const int col = c0 + ch * 16;
    if (PAIR) {
      if (nb == 2) {
        tmem_ld16x4(tb[0] + col, tb[0] + BN + col, tb[1] + col, tb[1] + BN + col, v[0], v[1],
                    v[2], v[3]);
      } else {
        tmem_ld16x2(tb[0] + col, tb[0] + BN + col, v[0], v[1]);
      }
    } else {
      if (nb == 4)
        tmem_ld16x4(tb[0] + col, tb[1] + col, tb[2] + col, tb[3] + col, v[0], v[1], v[2], v[3]);
      else if (nb >= 2)
        tmem_ld16x2(tb[0] + col, tb[1] + col, v[0], v[1]);
      else
        tmem_ld16(tb[0] + col, v[0]);
      if (nb == 3) tmem_ld16(tb[2] + col, v[2]);
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      if (b >= nb) break;
      const int gk = kbi + b;
      const float sw_g = sb[MAX_KB * BN + 2 * gk];
      const float sw_u = sb[MAX_KB * BN + 2 * gk + 1];
      const float* ts = sb + gk * BN + ch * 16 + c0;
      const float* pg = PAIR ? v[2 * b] : v[b];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float sa = ts[i];
        g[ch * 16 + i] = fmaf(pg[i], sw_g * sa, g[ch * 16 + i]);
        if (PAIR) u[ch * 16 + i] = fmaf(v[2 * b + 1][i], sw_u * sa, u[ch * 16 + i]);
      }
    }
  }
  tc_fence_before();
  __syncwarp();
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    if (b >= nb) break;
    if (lane == 0) mbar_arrive(&sm.tempty[acc]);
    if (++acc == C::NACC) { acc = 0; aphase ^= 1; }
  }
  return nb;
}

template <int BN, bool DET>
__device__ void run_epilogue(const GemmParams& p, Smem<BN>& sm, uint32_t tmem_base) {
  using C = Cfg<BN>;
  constexpr int COLS = C::COLS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ew = warp - C::FIRST_EPI_WARP;    // epilogue warp 0..7
  const int grp = ew / C::GROUP_WARPS;        // epilogue group (takes every NGROUPS-th unit)
  const int gw = ew - grp * C::GROUP_WARPS;   // warp within the group
  const int gtid = gw * 32 + lane;            // thread within the group
  const int quad = warp & 3;            // TMEM lane quadrant this warp may access
  const int half = gw >> 2;             // column group of this warp (groups of eight)
  const int row = quad * 32 + lane;     // output feature within the tile
  const int c0 = half * COLS;
  const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
  // named barriers of this group: all its threads, then one per column half
  const int bar_grp = 1 + grp * 3;
  int us = 0, acc = 0, steps = 0, seq = 0;
  uint32_t uphase = 0, aphase = 0;
  SigState sg;
  float* const sb = sm.sc + grp * C::SC_FLOATS;  // this group's per-unit scale staging
  const int G_L = p.L / 128, G_I = p.I / 128;

  for (;;) {
    if (!mbar_wait(&sm.ufull[us], uphase, sm.abort_flag, p.err, p.timeout)) return;
    const UnitInfo info = sm.ring[us];
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.uempty[us]);
    if (++us == C::US) { us = 0; uphase ^= 1; }
    if (info.task < 0) {
      signal_done<BN>(p, sm, sg, nullptr, grp, gw, lane);  // releases the group's signaller
      return;
    }
    const GemmTask& T = p.task[info.task];
    const int kind = T.kind;
    const bool pair = T.pair != 0;
    if (C::NGROUPS > 1 && (seq++ % C::NGROUPS) != grp) {
      // the other group's unit: step past the accumulator slots the MMA issuer fills for
      // it (one per promotion group, one for a whole-K unit, none for a norm unit)
      acc += kind == TASK_NORM ? 0 : (T.kpg > 0 ? (info.kb1 - info.kb0) / T.kpg : 1);
      while (acc >= C::NACC) {
        acc -= C::NACC;
        aphase ^= 1;
      }
      continue;
    }

    if (kind == TASK_NORM) {
      // RMSNorm of one token row (unit rows = 1): fp32 statistic on the fp32 combine,
      // gamma applied, rounded once to bf16 as the output GEMM's token operand.  The
      // epilogue threads split the row; each loads its float4s before using them.
      const size_t t = static_cast<size_t>(info.row0);
      const float4* rv = reinterpret_cast<const float4*>(p.r + t * p.L);
      // the combined row: r (added into by the routed L2 units), or the token's topk
      // weighted slots summed in choice order (deterministic combine)
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
      constexpr int PER = 8;  // float4s per thread held in registers
      const uint2* gg = reinterpret_cast<const uint2*>(p.gamma);
      float4 v[PER];
      uint2 gv[PER];  // gamma, loaded together with the row
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int c = gtid + i * C::GROUP_THREADS;
        v[i] = c < n4 ? row4(c) : make_float4(0.f, 0.f, 0.f, 0.f);
        gv[i] = c < n4 ? __ldg(gg + c) : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < PER; ++i) ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z +
                                         v[i].w * v[i].w;
      for (int c = gtid + PER * C::GROUP_THREADS; c < n4; c += C::GROUP_THREADS) {  // wide rows
        const float4 w = row4(c);
        ss += w.x * w.x + w.y * w.y + w.z * w.z + w.w * w.w;
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
      if (lane == 0) sm.red[ew * COLS] = ss;  // the first entry of this warp's own row
      named_bar_sync(bar_grp, C::GROUP_THREADS);
      float tot = 0.f;
      for (int w = 0; w < C::GROUP_WARPS; ++w) tot += sm.red[(grp * C::GROUP_WARPS + w) * COLS];
      const float inv = rsqrtf(tot / static_cast<float>(p.L) + p.eps);
      uint2* nn = reinterpret_cast<uint2*>(p.nrm + t * p.L);
      auto emit = [&](int c, const float4& x, const uint2 graw) {
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
      };
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int c = gtid + i * C::GROUP_THREADS;
        if (c < n4) emit(c, v[i], gv[i]);
      }
      for (int c = gtid + PER * C::GROUP_THREADS; c < n4; c += C::GROUP_THREADS)
        emit(c, row4(c), __ldg(gg + c));
      if constexpr (!DET) {
        // the row has been read (by this thread, the same elements): zero it for the next
        // forward's combine
        if (p.zero_r) {
          float4* rw = reinterpret_cast<float4*>(p.r + t * p.L);
          for (int c = gtid; c < n4; c += C::GROUP_THREADS) rw[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      named_bar_sync(bar_grp, C::GROUP_THREADS);  // sm.red is reused by the next unit
      signal_done<BN>(p, sm, sg, p.norm_done + info.dep_idx, grp, gw, lane);
      continue;
    }

    float g[COLS], u[COLS];
#pragma unroll
    for (int j = 0; j < COLS; ++j) { g[j] = 0.f; u[j] = 0.f; }

    if (T.kpg > 0) {
      // Stage this unit's scales in shared memory once: token group scales [group][column]
      // and the weight block scale(s) per 128-wide K group.  The group's staging buffer is
      // rewritten only after every thread of the group has finished its previous unit.
      const float* tok_scale = kind == TASK_ROUTED_L1 ? p.zsT : p.asT;
      named_bar_sync(bar_grp, C::GROUP_THREADS);
      const int nkb = (info.kb1 - info.kb0) / T.kpg;  // promotion groups of this unit
      const int g0 = info.kb0 / T.kpg;
      const int etid = gtid;
      for (int i = etid; i < nkb * BN; i += C::GROUP_THREADS) {
        const int kbi = i / BN, j = i - kbi * BN;
        sb[i] = j < info.rows
                    ? __ldcg(tok_scale + static_cast<size_t>(g0 + kbi) * p.cap + info.row0 + j)
                    : 0.f;
      }
      for (int kbi = etid; kbi < nkb; kbi += C::GROUP_THREADS) {
        const int kb = g0 + kbi;
        float a, b = 0.f;
        if (kind == TASK_ROUTED_L1) {
          const size_t rb = static_cast<size_t>(info.e) * (2 * G_I);
          a = __ldg(p.w13_s + (rb + info.ftile) * G_L + kb);
          b = __ldg(p.w13_s + (rb + G_I + info.ftile) * G_L + kb);
        } else {
          // one 128-row block, or two consecutive ones (paired units)
          const size_t rb = static_cast<size_t>(info.e) * G_L + info.ftile * T.a_rb_step;
          a = __ldg(p.w2_s + rb * G_I + kb);
          if (pair) b = __ldg(p.w2_s + (rb + 1) * G_I + kb);
        }
        sb[MAX_KB * BN + 2 * kbi] = a;
        sb[MAX_KB * BN + 2 * kbi + 1] = b;
      }
      if (kind == TASK_ROUTED_L2) {  // combine targets of each column
        for (int j = etid; j < BN; j += C::GROUP_THREADS) {
          const int pp = info.row0 + j;
          sb[MAX_KB * BN + 2 * MAX_KB + j] =
              __int_as_float(j < info.rows ? __ldg(p.gidx + pp) : 0);
          sb[MAX_KB * BN + 2 * MAX_KB + BN + j] = j < info.rows ? __ldg(p.wperm + pp) : 0.f;
        }
      }
      named_bar_sync(bar_grp, C::GROUP_THREADS);
      // Promote completed groups in batches: wait for up to NB slots, load them under one
      // TMEM wait, then scale-and-add, so the per-group latency chain is paid once per batch.
      for (int kbi = 0; kbi < nkb;) {
        const int left = nkb - kbi;
        int nb;
        if (pair)
          nb = promote_batch<BN, COLS, 2, true>(left, kbi, sb, g, u, sm, tmem_base, lane_base, c0,
                                                acc, aphase, p);
        else
          nb = promote_batch<BN, COLS, 4, false>(left, kbi, sb, g, u, sm, tmem_base, lane_base,
                                                 c0, acc, aphase, p);
        if (nb == 0) return;  // a bounded wait expired
        kbi += nb;
        if (ew == 0 && lane == 0) trace_mark(p, 2, steps++);
      }
    } else {
      if (!mbar_wait(&sm.tfull[acc], aphase, sm.abort_flag, p.err, p.timeout)) return;
      tc_fence_after();
      const uint32_t tb = tmem_base + lane_base + static_cast<uint32_t>(acc * C::SLOT_COLS);
#pragma unroll
      for (int ch = 0; ch < COLS / 16; ++ch) {
        if (pair)
          tmem_ld16x2(tb + c0 + ch * 16, tb + BN + c0 + ch * 16, g + ch * 16, u + ch * 16);
        else
          tmem_ld16(tb + c0 + ch * 16, g + ch * 16);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.tempty[acc]);
      if (++acc == C::NACC) { acc = 0; aphase ^= 1; }
      if (ew == 0 && lane == 0) trace_mark(p, 2, steps++);
    }

    // ---- split-K / stream-K: publish the partial; the last arriving contributor sums
    // all contributors' partials in a fixed order (deterministic)
    if (info.ncontrib > 1) {
      const int parts = pair ? 2 : 1;
      const size_t tile_floats = static_cast<size_t>(parts) * BN * 128;
      const size_t own =
          T.streamk ? static_cast<size_t>(info.wslot)
                    : static_cast<size_t>(info.tile_id - T.ws_tile_base) * info.ncontrib +
                          info.split;
      float* mine = p.ws + T.ws_off + own * tile_floats;
#pragma unroll
      for (int j = 0; j < COLS; ++j) {
        __stcg(mine + static_cast<size_t>(c0 + j) * 128 + row, g[j]);
        if (pair) __stcg(mine + static_cast<size_t>(BN + c0 + j) * 128 + row, u[j]);
      }
      __threadfence();
      named_bar_sync(bar_grp, C::GROUP_THREADS);
      if (gw == 0 && lane == 0) {
        const int old = atomicAdd(p.cnt + info.tile_id, 1);
        const int last = old == info.ncontrib - 1;
        if (last) p.cnt[info.tile_id] = 0;
        sm.last_flag[grp] = last;
      }
      named_bar_sync(bar_grp, C::GROUP_THREADS);
      if (!sm.last_flag[grp]) continue;
      __threadfence();
      // contributor s's partial: this thread's row of the part's first column
      auto part = [&](int s) -> const float* {
        const size_t idx =
            T.streamk ? static_cast<size_t>(sk_slot(T.sk_total, T.sk_grid, T.kb_total,
                                                    info.cfirst + s,
                                                    info.tile_id - T.ws_tile_base))
                      : static_cast<size_t>(info.tile_id - T.ws_tile_base) * info.ncontrib + s;
        return p.ws + T.ws_off + idx * tile_floats + static_cast<size_t>(c0) * 128 + row;
      };
#pragma unroll
      for (int j = 0; j < COLS; ++j) { g[j] = 0.f; u[j] = 0.f; }
      // The partials are added in contributor order 0, 1, ... whatever the batching.  With
      // few columns per thread the loads of several contributors are issued before any of
      // them is added, so their L2 round trips overlap instead of forming a chain (a tile
      // split ten ways otherwise pays ten round trips at the end of the launch).
      int s = 0;
      if constexpr (COLS <= 16) {
        // paired tiles: two contributors per batch (both parts); single tiles: four
        const int nb = pair ? 2 : 4;
        for (; s + nb <= info.ncontrib; s += nb) {
          const float* pa = part(s);
          const float* pb = part(s + 1);
          const float* pc = pair ? pa + static_cast<size_t>(BN) * 128 : part(s + 2);
          const float* pd = pair ? pb + static_cast<size_t>(BN) * 128 : part(s + 3);
          float va[COLS], vb[COLS], vc[COLS], vd[COLS];
#pragma unroll
          for (int j = 0; j < COLS; ++j) {
            va[j] = __ldcg(pa + static_cast<size_t>(j) * 128);
            vb[j] = __ldcg(pb + static_cast<size_t>(j) * 128);
            vc[j] = __ldcg(pc + static_cast<size_t>(j) * 128);
            vd[j] = __ldcg(pd + static_cast<size_t>(j) * 128);
          }
          if (pair) {
#pragma unroll
            for (int j = 0; j < COLS; ++j) {
              g[j] = (g[j] + va[j]) + vb[j];
              u[j] = (u[j] + vc[j]) + vd[j];
            }
          } else {
#pragma unroll
            for (int j = 0; j < COLS; ++j) g[j] = (((g[j] + va[j]) + vb[j]) + vc[j]) + vd[j];
          }
        }
      }
      for (; s < info.ncontrib; ++s) {
        const float* ps = part(s);
#pragma unroll
        for (int j = 0; j < COLS; ++j) {
          g[j] += __ldcg(ps + static_cast<size_t>(j) * 128);
          if (pair) u[j] += __ldcg(ps + static_cast<size_t>(BN + j) * 128);
        }
      }
    }

    // ---- fused epilogues
    if (kind == TASK_SHARED_L1) {
      __nv_bfloat16* dst = p.a_s + static_cast<size_t>(info.ftile) * 128 + row;
#pragma unroll
      for (int j = 0; j < COLS; ++j) {
        if (c0 + j < info.rows)
          dst[static_cast<size_t>(info.row0 + c0 + j) * p.Is] =
              __float2bfloat16_rn(silu_fast(g[j]) * u[j]);
      }
      if (p.sh_done != nullptr)
        signal_done<BN>(p, sm, sg, p.sh_done + info.dep_idx, grp, gw, lane);
    } else if (kind == TASK_PROJ) {
      // projection rows [0, L): the latent input (bf16); [L, L + E): router logits (fp32);
      // beyond: zero padding of the weight image, not stored
      const int f0 = info.arb * 128 + row;
#pragma unroll
      for (int j = 0; j < COLS; ++j) {
        if (c0 + j < info.rows) {
          const size_t t = static_cast<size_t>(info.row0 + c0 + j);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            if (h2 == 1 && !pair) break;
            const int f = f0 + 128 * h2;
            const float v = h2 ? u[j] : g[j];
            if (f < p.L)
              p.zp[t * p.L + f] = __float2bfloat16_rn(v);
            else if (f < p.L + p.E)
              p.lgp[t * p.E + (f - p.L)] = v;
          }
        }
      }
    } else if (kind == TASK_OUT) {
      // g: the unit's first 128 output features; u: the next 128 (paired units)
      __nv_bfloat16* dst = p.out + static_cast<size_t>(info.arb) * 128 + row;
#pragma unroll
      for (int j = 0; j < COLS; ++j) {
        if (c0 + j < info.rows) {
          __nv_bfloat16* o = dst + static_cast<size_t>(info.row0 + c0 + j) * p.H;
          o[0] = __float2bfloat16_rn(g[j]);
          if (pair) o[128] = __float2bfloat16_rn(u[j]);
        }
      }
    } else if (kind == TASK_ROUTED_L2) {
      // g: the unit's first 128 output rows; u: the next 128 (paired units)
      const int col = info.ftile * 128 * T.a_rb_step + row;
#pragma unroll
      for (int j = 0; j < COLS; ++j) {
        if (c0 + j < info.rows) {
          const int tok = __float_as_int(sb[MAX_KB * BN + 2 * MAX_KB + c0 + j]);
          const float wv = sb[MAX_KB * BN + 2 * MAX_KB + BN + c0 + j];
          if constexpr (DET) {  // this pair's weighted output, summed later in choice order
            float* y = p.yw + static_cast<size_t>(info.row0 + c0 + j) * p.L + col;
            y[0] = wv * g[j];
            if (pair) y[128] = wv * u[j];
          } else {
            float* y = p.r + static_cast<size_t>(tok) * p.L + col;
            atomicAdd(y, wv * g[j]);
            if (pair) atomicAdd(y + 128, wv * u[j]);
          }
        }
      }
      if (p.l2_done != nullptr) signal_done<BN>(p, sm, sg, p.l2_done, grp, gw, lane);
    } else {  // TASK_ROUTED_L1: SwiGLU, then e4m3 per 128 features of each token
      float* red = sm.red + ew * COLS;
#pragma unroll
      for (int j = 0; j < COLS; ++j) {
        g[j] = silu_fast(g[j]) * u[j];
        float a = fabsf(g[j]);
#pragma unroll
        for (int o = 16; o; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
        if (lane == 0) red[j] = a;
      }
      named_bar_sync(bar_grp + 1 + half, 128);
      const float* r0 = sm.red + (grp * C::GROUP_WARPS + half * 4) * COLS;
      uint8_t* dst = p.aq + static_cast<size_t>(info.ftile) * 128 + row;
#pragma unroll
      for (int j = 0; j < COLS; ++j) {
        const float amax = fmaxf(fmaxf(r0[j], r0[COLS + j]), fmaxf(r0[2 * COLS + j],
                                                                   r0[3 * COLS + j]));
        // s = fp32(amax / 448) exactly (quotient by the correctly rounded 1/448)
        const float s = amax == 0.f ? 1.0f : quot_rn(amax, 448.0f, 1.0f / 448.0f);
        const float inv = rcp_nr(s);
        if (c0 + j < info.rows) {
          const size_t pp = static_cast<size_t>(info.row0 + c0 + j);
          const uint8_t code = f32_to_e4m3(quot_rn(g[j], s, inv));
          dst[pp * p.I] = code;
          if (p.aqb != nullptr)
            p.aqb[pp * p.I + static_cast<size_t>(info.ftile) * 128 + row] =
                __float2bfloat16_rn(e4m3_to_f32(code));
          if (quad == 0 && lane == 0) p.asT[static_cast<size_t>(info.ftile) * p.cap + pp] = s;
        }
      }
      named_bar_sync(bar_grp + 1 + half, 128);
      if (p.l1_done != nullptr)
        signal_done<BN>(p, sm, sg, p.l1_done + info.dep_idx, grp, gw, lane);
    }
  }
}

template <int BN, bool DET>
__global__ void __launch_bounds__(Cfg<BN>::THREADS, 1)
    gemm_kernel(const __grid_constant__ GemmParams p) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  Smem<BN> sm(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int a = 0; a < C::NACC; ++a) {
      mbar_init(&sm.tfull[a], 1);
      mbar_init(&sm.tempty[a], C::GROUP_WARPS);  // the warps of the group that owns the unit
    }
    for (int u = 0; u < C::US; ++u) {
      mbar_init(&sm.ufull[u], 1);
      mbar_init(&sm.uempty[u], 1 + C::EPI_WARPS);
    }
    for (int g = 0; g < Smem<BN>::NSIG; ++g) {
      mbar_init(&sm.sfull[g], C::GROUP_WARPS);
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
    tmem_alloc(sm.tmem_holder, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_holder;

  // Everything above touches only this CTA's resources, and the L2 prefetch below only
  // handle-owned weights that no kernel writes; inputs written by the previous kernels in
  // the stream are read only after the wait.  The routing kernels let this launch start
  // while they run, so the prefetch of routing-independent weights overlaps them.
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
    u0 = (lane == 0 && !p.task[0].streamk) ? atomicAdd(p.sched, 1) : 0;
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
  if (warp < C::FIRST_EPI_WARP) {
    regs_dec<C::REGS_CTRL>();
    if (warp == 0) {
      if (lane == 0) run_producer<BN>(p, sm, s_tile_off, s_off, u0);
    } else if (warp == 1) {
      if (lane == 0) run_mma<BN>(p, sm, tmem_base);
    } else if (warp - C::SIGNAL_WARP < C::NGROUPS && lane == 0) {
      run_signaller<BN>(p, sm, warp - C::SIGNAL_WARP);
    }
  } else {
    regs_inc<C::REGS_EPI>();
    run_epilogue<BN, DET>(p, sm, tmem_base);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <int BN>
cudaError_t launch_bn(const GemmParams& p, int grid, cudaStream_t s, bool pdl) {
  using C = Cfg<BN>;
  const int smem = Smem<BN>::bytes();
  // the deterministic combine is a separate instantiation (no code in the default one)
  const bool det = p.yw != nullptr;
  cudaError_t e = cudaFuncSetAttribute(det ? gemm_kernel<BN, true> : gemm_kernel<BN, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return det ? cudaLaunchKernelEx(&cfg, gemm_kernel<BN, true>, p)
             : cudaLaunchKernelEx(&cfg, gemm_kernel<BN, false>, p);
}

}  // namespace

// dynamic shared memory plus the producer's static offset tables
static_assert(Smem<16>::bytes() + 2 * (MAX_E + 1) * 4 <= 227 * 1024, "shared memory budget");
static_assert(Smem<32>::bytes() + 2 * (MAX_E + 1) * 4 <= 227 * 1024, "shared memory budget");
static_assert(Smem<64>::bytes() + 2 * (MAX_E + 1) * 4 <= 227 * 1024, "shared memory budget");
static_assert(Smem<128>::bytes() + 2 * (MAX_E + 1) * 4 <= 227 * 1024, "shared memory budget");

// Every instantiation must launch with the register count its hand-over was planned for.
bool gemm_regs_ok() {
  const void* k[] = {
      reinterpret_cast<const void*>(gemm_kernel<16, false>),
      reinterpret_cast<const void*>(gemm_kernel<16, true>),
      reinterpret_cast<const void*>(gemm_kernel<32, false>),
      reinterpret_cast<const void*>(gemm_kernel<32, true>),
      reinterpret_cast<const void*>(gemm_kernel<64, false>),
      reinterpret_cast<const void*>(gemm_kernel<64, true>),
      reinterpret_cast<const void*>(gemm_kernel<128, false>),
      reinterpret_cast<const void*>(gemm_kernel<128, true>)};
  for (const void* f : k) {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, f) != cudaSuccess || a.numRegs != Cfg<16>::LAUNCH_REGS)
      return false;
  }
  return true;
}

int gemm_smem_bytes(int bn) {
  switch (bn) {
    case 16: return Smem<16>::bytes();
    case 32: return Smem<32>::bytes();
    case 64: return Smem<64>::bytes();
    default: return Smem<128>::bytes();
  }
}

cudaError_t launch_gemm(const GemmParams& p, int bn, int grid, cudaStream_t s, bool pdl) {
  if (bn == 16) return launch_bn<16>(p, grid, s, pdl);
  if (bn == 32) return launch_bn<32>(p, grid, s, pdl);
  if (bn == 64) return launch_bn<64>(p, grid, s, pdl);
  if (bn == 128) return launch_bn<128>(p, grid, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace klt
