// Routing, latent activation quantisation, expert permutation and the RMSNorm step of the
// latent-MoE tail (sm_103a).
//
//  route_quant_kernel  top-k + softmax over the selected logits per token, e4m3 per-128
//                      quantisation of z, zeroing of the fp32 combine buffer r.
//  perm_hist_kernel    per-block expert histogram of the (token, choice) pairs.
//  perm_scatter_kernel stable counting-sort scatter: cnt/off/tile_off, gidx/slot/pos.
//  perm_gather_kernel  gather of each pair's quantised latent row into expert order (the
//                      routed L1 GEMM reads it with plain TMA tiles).
//  route_small_kernel  the three above in one launch for a small batch (one permutation
//                      block, e4m3 activations).
//  norm_kernel         RMSNorm of the routed combine with fp32 statistics on the fp32
//                      sum (tokenspeed PR 1062 commit notes: fp32-internal norm), gamma
//                      applied, rounded once to bf16 as the up-projection operand.
#include "klt_device.cuh"
#include "klt_internal.h"

namespace klt {

namespace {

__device__ __forceinline__ uint32_t ordered_key(float v) {
  uint32_t u = __float_as_uint(v);
  if ((u & 0x7FFFFFFFu) == 0) u = 0;  // -0 and +0 compare equal
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// e4m3 codes of one 128-column group held 4 columns per lane: s = amax / 448 (1 for an
// all-zero group), codes e4m3(v / s) with fp32(v / s) from the correctly rounded reciprocal
// (Markstein's correction).  Returns this lane's 4 codes, the first column in the low byte.
__device__ __forceinline__ uint32_t quant128_e4m3(float v0, float v1, float v2, float v3,
                                                  float& s_out) {
  float amax = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  const float s = amax == 0.f ? 1.0f : amax / 448.0f;
  const float inv = 1.0f / s;
  s_out = s;
  return f32x2_to_e4m3x2(quot_rn(v0, s, inv), quot_rn(v1, s, inv)) |
         (f32x2_to_e4m3x2(quot_rn(v2, s, inv), quot_rn(v3, s, inv)) << 16);
}

// Top-k of token t's logits with softmax over the selected ones, by one warp: the key is
// (ordered logit, inverted index), so the larger key wins and equal logits go to the lower
// expert index.  Lane j < k returns choice j's expert and weight.
__device__ __forceinline__ void route_token(const float* logits, int E, int k, int t, int lane,
                                            int& idx_out, float& wt_out) {
  const float* lg = logits + static_cast<size_t>(t) * E;
  constexpr int PER_LANE = MAX_E / 32;
  uint32_t keys[PER_LANE];
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) {
    const int e = lane + 32 * i;
    keys[i] = e < E ? ordered_key(__ldg(lg + e)) : 0u;
  }
  uint32_t taken = 0;  // bit i: entry i of this lane already selected
  int my_idx = 0;
  float my_val = 0.f;
  for (int j = 0; j < k; ++j) {
    unsigned long long best = 0ull;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !(taken >> i & 1u)) {
        const unsigned long long kk =
            (static_cast<unsigned long long>(keys[i]) << 32) | (0xFFFFFFFFu - e);
        best = kk > best ? kk : best;
      }
    }
    // the warp's largest 64-bit key: the largest high word, then the largest low word
    // among the lanes holding it
    const uint32_t hi = static_cast<uint32_t>(best >> 32);
    const uint32_t top = __reduce_max_sync(0xFFFFFFFFu, hi);
    const uint32_t lo =
        __reduce_max_sync(0xFFFFFFFFu, hi == top ? static_cast<uint32_t>(best) : 0u);
    const int e = static_cast<int>(0xFFFFFFFFu - lo);
    if ((e & 31) == lane) taken |= 1u << (e >> 5);
    if (lane == j) {
      my_idx = e;
      my_val = __ldg(lg + e);
    }
  }
  const float vmax = __shfl_sync(0xFFFFFFFFu, my_val, 0);
  const float ex = lane < k ? expf(my_val - vmax) : 0.f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
  idx_out = my_idx;
  wt_out = ex / sum;
}

// Quantisation of 128-column group g of token t's latent row (4 columns per lane, already
// loaded into `raw`).
__device__ __forceinline__ void quant_group(const RouteParams& p, int t, int g, uint2 raw,
                                            int lane) {
  const int G = p.L / 128;
  const __nv_bfloat162 b01 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
  const __nv_bfloat162 b23 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
  const float v0 = __low2float(b01), v1 = __high2float(b01);
  const float v2 = __low2float(b23), v3 = __high2float(b23);
  float amax = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
  uint32_t q;
  if (p.bs == BS_NV4) {
    // NVFP4: per 16 columns (4 lanes) s = e4m3(amax / 6), codes e2m1(v / s) (a zero scale
    // gives zero codes); quotients correctly rounded in fp32; two codes per byte, the even
    // column in the low nibble
#pragma unroll
    for (int o = 2; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    // correctly rounded quotients from correctly rounded reciprocals (Markstein's
    // correction, as in the GEMM epilogues): fp32(amax / 6) and fp32(v / s)
    const uint8_t sc = f32_to_e4m3(quot_rn(amax, 6.0f, 1.0f / 6.0f));
    const float s = e4m3_to_f32(sc);
    uint32_t c = 0;
    if (s != 0.f) {
      const float inv = 1.0f / s;
      c = f32x8_to_e2m1x8(quot_rn(v0, s, inv), quot_rn(v1, s, inv), quot_rn(v2, s, inv),
                          quot_rn(v3, s, inv), 0.f, 0.f, 0.f, 0.f);
    }
    if ((lane & 3) == 0) p.zsx[static_cast<size_t>(t) * (p.L / 16) + g * 8 + (lane >> 2)] = sc;
    *reinterpret_cast<uint16_t*>(p.zq + static_cast<size_t>(t) * (p.L / 2) + g * 64 +
                                 lane * 2) = static_cast<uint16_t>(c);
    return;
  }
  if (p.bs == BS_MX8) {
    // MX: one power-of-two scale per 32 columns (8 lanes): 2^(floor(log2 amax) - 8); the
    // quotient by a power of two is exact, so the codes equal e4m3(v / scale)
#pragma unroll
    for (int o = 4; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const int e = mx_exponent(amax);
    const float inv = pow2_exact(-e);
    q = static_cast<uint32_t>(f32_to_e4m3(v0 * inv)) |
        (static_cast<uint32_t>(f32_to_e4m3(v1 * inv)) << 8) |
        (static_cast<uint32_t>(f32_to_e4m3(v2 * inv)) << 16) |
        (static_cast<uint32_t>(f32_to_e4m3(v3 * inv)) << 24);
    if ((lane & 7) == 0)
      p.zsx[static_cast<size_t>(t) * (p.L / 32) + g * 4 + (lane >> 3)] =
          static_cast<uint8_t>(e + 127);
  } else {
    float s;
    q = quant128_e4m3(v0, v1, v2, v3, s);
    if (lane == 0) p.zs[static_cast<size_t>(t) * G + g] = s;
  }
  *reinterpret_cast<uint32_t*>(p.zq + static_cast<size_t>(t) * p.L + g * 128 + lane * 4) = q;
}

// Warp w handles token t = w / (P + 1), P = ceil(G / ROUTE_QG): part 0 routes the token,
// part j + 1 quantises its 128-column groups [j * ROUTE_QG, (j + 1) * ROUTE_QG) of z.  The
// combine buffer r the routed L2 units add into was zeroed by the previous forward's norm.
__global__ void __launch_bounds__(32 * ROUTE_WARPS)
    route_quant_kernel(const RouteParams p) {
  pdl_trigger();  // dependents may launch now; they wait for this grid before reading
  pdl_wait();
  const int lane = lane_id();
  if (blockIdx.x == 0 && threadIdx.x < p.nsched) p.sched[threadIdx.x] = 0;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
       i < p.zero_n; i += static_cast<long long>(gridDim.x) * blockDim.x)
    p.zero_buf[i] = 0;
  const int G = p.L / 128;
  const int P = (G + ROUTE_QG - 1) / ROUTE_QG;
  const long long w = static_cast<long long>(blockIdx.x) * ROUTE_WARPS + (threadIdx.x >> 5);
  const int t = static_cast<int>(w / (P + 1));
  const int part = static_cast<int>(w - static_cast<long long>(t) * (P + 1));
  if (t >= p.M) return;

  if (part == 0) {
    int idx;
    float wt;
    route_token(p.logits, p.E, p.k, t, lane, idx, wt);
    if (lane < p.k) {
      p.ids[static_cast<size_t>(t) * p.k + lane] = idx;
      p.wts[static_cast<size_t>(t) * p.k + lane] = wt;
    }
    return;
  }

  // ---- quantisation of up to QG consecutive 128-column groups: their loads are issued
  // together, so a warp has several DRAM round trips in flight
  const int g0 = (part - 1) * ROUTE_QG;
  uint2 raw[ROUTE_QG];
#pragma unroll
  for (int j = 0; j < ROUTE_QG; ++j)
    if (g0 + j < G)
      raw[j] = *reinterpret_cast<const uint2*>(p.z + static_cast<size_t>(t) * p.L +
                                                (g0 + j) * 128 + lane * 4);
#pragma unroll
  for (int j = 0; j < ROUTE_QG; ++j)
    if (g0 + j < G) quant_group(p, t, g0 + j, raw[j], lane);
}

__global__ void __launch_bounds__(PERM_BLOCK) perm_hist_kernel(const PermParams p) {
  __shared__ int hist[MAX_E];
  pdl_trigger();  // dependents may launch now; they wait for this grid before reading
  pdl_wait();
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int i = blockIdx.x * PERM_BLOCK + threadIdx.x;
  if (i < p.M * p.k) atomicAdd(&hist[p.ids[i]], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < p.E; e += blockDim.x)
    p.hist[blockIdx.x * p.E + e] = hist[e];
}

__global__ void __launch_bounds__(PERM_BLOCK) perm_scatter_kernel(const PermParams p) {
  __shared__ int warp_cnt[PERM_BLOCK / 32][MAX_E];
  __shared__ int base[MAX_E];
  __shared__ int total[MAX_E];
  __shared__ int tiles[MAX_E];
  pdl_trigger();  // dependents may launch now; they wait for this grid before reading
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int Mk = p.M * p.k;
  for (int c = tid; c < (PERM_BLOCK / 32) * MAX_E; c += PERM_BLOCK)
    (&warp_cnt[0][0])[c] = 0;
  // expert totals and the count of this expert's pairs in earlier blocks (a single block
  // counts its own pairs and needs no histogram pass)
  if (p.nblocks == 1) {
    if (tid < p.E) total[tid] = 0;
    __syncthreads();
    if (tid < Mk) atomicAdd(&total[p.ids[tid]], 1);
    __syncthreads();
    if (tid < p.E) {
      base[tid] = 0;
      tiles[tid] = (total[tid] + p.bn - 1) / p.bn;
    }
  } else if (tid < p.E) {
    int tot = 0, pre = 0;
    for (int b = 0; b < p.nblocks; ++b) {
      const int h = p.hist[b * p.E + tid];
      tot += h;
      if (b < static_cast<int>(blockIdx.x)) pre += h;
    }
    total[tid] = tot;
    base[tid] = pre;
    tiles[tid] = (tot + p.bn - 1) / p.bn;
  }
  __syncthreads();
  if (tid == 0) {  // exclusive scans over experts (E <= 256)
    int acc = 0, tacc = 0;
    for (int e = 0; e < p.E; ++e) {
      const int c = total[e], tc = tiles[e];
      total[e] = acc;  // now the expert offset
      tiles[e] = tacc;
      acc += c;
      tacc += tc;
      if (blockIdx.x == 0) {
        p.cnt[e] = c;
        p.off[e] = total[e];
        p.tile_off[e] = tiles[e];
      }
    }
    if (blockIdx.x == 0) {
      p.off[p.E] = acc;
      p.tile_off[p.E] = tacc;
    }
  }
  __syncthreads();
  if (tid < p.E) base[tid] += total[tid];

  // rank inside the warp among pairs of the same expert (lower lane = lower pair index)
  const int i = blockIdx.x * PERM_BLOCK + tid;
  const int e = i < Mk ? p.ids[i] : -1 - lane;  // inactive lanes get unique keys
  const unsigned same = __match_any_sync(0xFFFFFFFFu, e);
  const int rank = __popc(same & ((1u << lane) - 1u));
  if (e >= 0 && rank == 0) warp_cnt[w][e] = __popc(same);
  __syncthreads();
  if (tid < p.E) {  // exclusive scan over warps, per expert
    int acc = 0;
    for (int ww = 0; ww < PERM_BLOCK / 32; ++ww) {
      const int c = warp_cnt[ww][tid];
      warp_cnt[ww][tid] = acc;
      acc += c;
    }
  }
  __syncthreads();
  if (e >= 0) {
    const int pp = base[e] + warp_cnt[w][e] + rank;
    p.gidx[pp] = i / p.k;
    p.slot[pp] = i;
    p.pos[i] = pp;
    p.wperm[pp] = p.wts[i];
  }
}

// Gather of each pair's quantised latent row (and its scales, transposed to [group, pair])
// into pair order, so the routed L1 GEMM streams an expert's token rows as plain tiles.
// One thread per 16-byte chunk.
__global__ void __launch_bounds__(256) perm_gather_kernel(const PermParams p) {
  pdl_trigger();  // dependents may launch now; they wait for this grid before reading
  pdl_wait();
  const int G = p.L / 128;
  const int row16 = p.zrow / 16;  // 16-byte chunks of a quantised latent row
  const long long Mk = static_cast<long long>(p.M) * p.k;
  const long long c = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
  if (c < Mk * row16) {
    const int pp = static_cast<int>(c / row16);
    const int ch = static_cast<int>(c - static_cast<long long>(pp) * row16);
    const int t = __ldg(p.gidx + pp);
    const uint4 v = reinterpret_cast<const uint4*>(p.zq + static_cast<size_t>(t) * p.zrow)[ch];
    if (p.zqb_perm == nullptr) {
      reinterpret_cast<uint4*>(p.zq_perm + static_cast<size_t>(pp) * p.zrow)[ch] = v;
    } else {  // exact bf16 image of every e4m3 code (bf16-operand layers)
      const uint8_t* b = reinterpret_cast<const uint8_t*>(&v);
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(e4m3_to_f32(b[2 * i]),
                                                       e4m3_to_f32(b[2 * i + 1]));
        o[i] = *reinterpret_cast<const uint32_t*>(&h);
      }
      uint4* dst = reinterpret_cast<uint4*>(p.zqb_perm + static_cast<size_t>(pp) * p.L +
                                            static_cast<size_t>(ch) * 16);
      dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
      dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
  }
  if (p.zsf_t == nullptr && c < Mk * G) {
    const int pp = static_cast<int>(c / G);
    const int g = static_cast<int>(c - static_cast<long long>(pp) * G);
    p.zsT[static_cast<size_t>(g) * p.cap + pp] =
        p.zs[static_cast<size_t>(__ldg(p.gidx + pp)) * G + g];
  }
  // Block-scaled layers: the token scale tiles of every routed tile (one 4-byte word per
  // tile row and tile a); rows past the tile's pairs get a unit scale (their products are
  // never stored)
  const int nsc = p.L / p.sf_group;  // scale bytes per row
  const int NA = nsc / 4;            // scale tiles per routed tile
  if (p.zsf_t != nullptr && c < static_cast<long long>(p.sf_tiles) * 128 * NA) {
    const int tile = static_cast<int>(c / (128LL * NA));
    const int rem = static_cast<int>(c - static_cast<long long>(tile) * 128 * NA);
    const int kb = rem / 128, r = rem - (rem / 128) * 128;
    if (tile < p.tile_off[p.E]) {
      int lo = 0, hi = p.E - 1;  // largest e with tile_off[e] <= tile
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(p.tile_off + mid) <= tile) lo = mid; else hi = mid - 1;
      }
      const int pp = __ldg(p.off + lo) + (tile - __ldg(p.tile_off + lo)) * p.bn + r;
      // unit scale: UE8M0 127 (MX) or e4m3 1.0 (NVFP4)
      uint32_t word = p.sf_group == 32 ? 0x7F7F7F7Fu : 0x38383838u;
      if (pp < __ldg(p.off + lo + 1))
        word = *reinterpret_cast<const uint32_t*>(
            p.zsx + static_cast<size_t>(__ldg(p.gidx + pp)) * nsc + 4 * kb);
      *reinterpret_cast<uint32_t*>(p.zsf_t + (static_cast<size_t>(tile) * NA + kb) * 512 +
                                   (r & 31) * 16 + 4 * (r >> 5)) = word;
    }
  }
}

// Routing, quantisation and permutation of a small batch (M·k <= SMALL_PAIRS pairs, one
// permutation block) in one launch instead of three.  Every block routes all M tokens and
// counting-sorts the pairs in shared memory, with the arithmetic and the stable order of
// route_quant_kernel and perm_scatter_kernel; block 0 publishes the routing arrays.  Then
// warp w of the grid quantises QG consecutive 128-column groups of one pair's latent row
// (item w = pair * P + part, P = ceil(G / QG)) straight into expert order (zq_perm or its
// bf16 image, zsT); the pair that is its token's choice 0 also writes the token-order zq
// and zs.  Only e4m3 activations (per-128 fp32 scales) take this path.
__global__ void __launch_bounds__(SMALL_THREADS)
    route_small_kernel(const RouteParams rp, const PermParams p) {
  constexpr int NW = SMALL_THREADS / 32;  // warps per block
  constexpr int PW = SMALL_PAIRS / 32;    // warps holding a pair
  __shared__ int s_ids[SMALL_PAIRS];
  __shared__ float s_wts[SMALL_PAIRS];
  __shared__ int s_gidx[SMALL_PAIRS];
  __shared__ int s_slot[SMALL_PAIRS];
  __shared__ int warp_cnt[PW][MAX_E];
  __shared__ int total[MAX_E];
  pdl_trigger();  // dependents may launch now; they wait for this grid before reading
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int E = rp.E, k = rp.k, Mk = rp.M * rp.k;
  const bool pub = blockIdx.x == 0;
  if (pub && tid < rp.nsched) rp.sched[tid] = 0;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + tid; i < rp.zero_n;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    rp.zero_buf[i] = 0;
  for (int c = tid; c < PW * MAX_E; c += SMALL_THREADS) (&warp_cnt[0][0])[c] = 0;
  if (tid < E) total[tid] = 0;

  // ---- top-k of every token (warp w: tokens w, w + NW, ...)
  for (int t = w; t < rp.M; t += NW) {
    int idx;
    float wt;
    route_token(rp.logits, E, k, t, lane, idx, wt);
    if (lane < k) {
      s_ids[t * k + lane] = idx;
      s_wts[t * k + lane] = wt;
      if (pub) {
        rp.ids[static_cast<size_t>(t) * k + lane] = idx;
        rp.wts[static_cast<size_t>(t) * k + lane] = wt;
      }
    }
  }
  __syncthreads();

  // ---- stable counting sort of the pairs by expert
  if (tid < Mk) atomicAdd(&total[s_ids[tid]], 1);
  __syncthreads();
  if (w == 0) {  // exclusive scans over experts, 32 at a time
    int acc = 0, tacc = 0;
    for (int b = 0; b < E; b += 32) {
      const int e = b + lane;
      const int c = e < E ? total[e] : 0, tc = (c + p.bn - 1) / p.bn;
      int ic = c, it = tc;  // inclusive scans across the lanes
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xFFFFFFFFu, ic, o);
        const int y = __shfl_up_sync(0xFFFFFFFFu, it, o);
        if (lane >= o) {
          ic += x;
          it += y;
        }
      }
      if (e < E) {
        total[e] = acc + ic - c;  // now the expert offset
        if (pub) {
          p.cnt[e] = c;
          p.off[e] = acc + ic - c;
          p.tile_off[e] = tacc + it - tc;
        }
      }
      acc += __shfl_sync(0xFFFFFFFFu, ic, 31);
      tacc += __shfl_sync(0xFFFFFFFFu, it, 31);
    }
    if (pub && lane == 0) {
      p.off[E] = acc;
      p.tile_off[E] = tacc;
    }
  }
  // rank inside the warp among pairs of the same expert (lower lane = lower pair index)
  const int e = tid < Mk ? s_ids[tid] : -1 - lane;  // inactive lanes get unique keys
  const unsigned same = __match_any_sync(0xFFFFFFFFu, e);
  const int rank = __popc(same & ((1u << lane) - 1u));
  if (e >= 0 && rank == 0) warp_cnt[w][e] = __popc(same);  // e >= 0 only in warps < PW
  __syncthreads();
  if (tid < E) {  // exclusive scan over warps, per expert
    int acc = 0;
    for (int ww = 0; ww < PW; ++ww) {
      const int c = warp_cnt[ww][tid];
      warp_cnt[ww][tid] = acc;
      acc += c;
    }
  }
  __syncthreads();
  if (e >= 0) {
    const int pp = total[e] + warp_cnt[w][e] + rank;
    s_gidx[pp] = tid / k;
    s_slot[pp] = tid;
    if (pub) {
      p.gidx[pp] = tid / k;
      p.slot[pp] = tid;
      p.pos[tid] = pp;
      p.wperm[pp] = s_wts[tid];
    }
  }
  __syncthreads();

  // ---- quantisation into expert order
  const int G = rp.L / 128;
  const int P = (G + ROUTE_QG - 1) / ROUTE_QG;
  const long long item = static_cast<long long>(blockIdx.x) * NW + w;
  if (item >= static_cast<long long>(Mk) * P) return;
  const int pp = static_cast<int>(item / P);
  const int g0 = static_cast<int>(item - static_cast<long long>(pp) * P) * ROUTE_QG;
  const int t = s_gidx[pp];
  const bool first = s_slot[pp] % k == 0;  // the token's choice 0 writes token order
  uint2 raw[ROUTE_QG];
#pragma unroll
  for (int j = 0; j < ROUTE_QG; ++j)
    if (g0 + j < G)
      raw[j] = *reinterpret_cast<const uint2*>(rp.z + static_cast<size_t>(t) * rp.L +
                                                (g0 + j) * 128 + lane * 4);
#pragma unroll
  for (int j = 0; j < ROUTE_QG; ++j) {
    const int g = g0 + j;
    if (g >= G) break;
    const __nv_bfloat162 b01 = *reinterpret_cast<const __nv_bfloat162*>(&raw[j].x);
    const __nv_bfloat162 b23 = *reinterpret_cast<const __nv_bfloat162*>(&raw[j].y);
    float sc;
    const uint32_t q = quant128_e4m3(__low2float(b01), __high2float(b01), __low2float(b23),
                                     __high2float(b23), sc);
    const size_t col = static_cast<size_t>(g) * 128 + lane * 4;
    if (p.zqb_perm == nullptr) {
      *reinterpret_cast<uint32_t*>(p.zq_perm + static_cast<size_t>(pp) * rp.L + col) = q;
    } else {  // exact bf16 image of every e4m3 code (bf16-operand layers)
      const __nv_bfloat162 h01 = __floats2bfloat162_rn(e4m3_to_f32(q & 0xFF),
                                                       e4m3_to_f32((q >> 8) & 0xFF));
      const __nv_bfloat162 h23 = __floats2bfloat162_rn(e4m3_to_f32((q >> 16) & 0xFF),
                                                       e4m3_to_f32(q >> 24));
      *reinterpret_cast<uint2*>(p.zqb_perm + static_cast<size_t>(pp) * rp.L + col) =
          make_uint2(*reinterpret_cast<const uint32_t*>(&h01),
                     *reinterpret_cast<const uint32_t*>(&h23));
    }
    if (lane == 0) p.zsT[static_cast<size_t>(g) * p.cap + pp] = sc;
    if (first) {
      *reinterpret_cast<uint32_t*>(rp.zq + static_cast<size_t>(t) * rp.L + col) = q;
      if (lane == 0) rp.zs[static_cast<size_t>(t) * G + g] = sc;
    }
  }
}

__global__ void __launch_bounds__(128) norm_kernel(const NormParams p) {
  __shared__ float red[4];
  pdl_trigger();  // dependents may launch now; they wait for this grid before reading
  pdl_wait();
  const int t = blockIdx.x;
  const float4* rr = reinterpret_cast<const float4*>(p.r + static_cast<size_t>(t) * p.L);
  float ss = 0.f;
  for (int c = threadIdx.x; c < p.L / 4; c += 128) {
    const float4 v = rr[c];
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  const float tot = red[0] + red[1] + red[2] + red[3];
  const float inv = rsqrtf(tot / static_cast<float>(p.L) + p.eps);
  const uint2* gg = reinterpret_cast<const uint2*>(p.gamma);
  uint2* nn = reinterpret_cast<uint2*>(p.n + static_cast<size_t>(t) * p.L);
  float4* rz = reinterpret_cast<float4*>(p.r) + static_cast<size_t>(t) * (p.L / 4);
  for (int c = threadIdx.x; c < p.L / 4; c += 128) {
    const float4 v = rr[c];
    if (p.zero_r) rz[c] = make_float4(0.f, 0.f, 0.f, 0.f);  // ready for the next forward
    const uint2 graw = gg[c];
    const __nv_bfloat162 g01 = *reinterpret_cast<const __nv_bfloat162*>(&graw.x);
    const __nv_bfloat162 g23 = *reinterpret_cast<const __nv_bfloat162*>(&graw.y);
    const __nv_bfloat162 o01 = __floats2bfloat162_rn(v.x * inv * __low2float(g01),
                                                     v.y * inv * __high2float(g01));
    const __nv_bfloat162 o23 = __floats2bfloat162_rn(v.z * inv * __low2float(g23),
                                                     v.w * inv * __high2float(g23));
    uint2 o;
    o.x = *reinterpret_cast<const uint32_t*>(&o01);
    o.y = *reinterpret_cast<const uint32_t*>(&o23);
    nn[c] = o;
  }
}

__global__ void __launch_bounds__(256)
    tile_relayout_kernel(const uint8_t* src, uint8_t* dst, long long rows, long long row_bytes) {
  const long long c16 = row_bytes / 16;
  const long long q = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
  if (q >= rows * c16) return;
  const long long row = q / c16, col = q - row * c16;
  const long long rb = row >> 7, r = row & 127, kb = col >> 3, ch = col & 7;
  const long long dst_off = (((rb * (row_bytes / 128)) + kb) * 128 + r) * 128 + ((ch ^ (r & 7)) * 16);
  *reinterpret_cast<uint4*>(dst + dst_off) =
      *reinterpret_cast<const uint4*>(src + row * row_bytes + col * 16);
}

// 16-byte output chunk q = 8 bf16 values of row r at K offset k0 (8 | k0, one scale block).
__global__ void __launch_bounds__(256)
    nvfp4_expand_kernel(const uint8_t* packed, const uint8_t* sb, uint8_t* dst, long long rows,
                        long long K) {
  const long long c16 = K / 8;
  const long long q = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
  if (q >= rows * c16) return;
  const long long row = q / c16, col = q - row * c16;
  const long long k0 = col * 8;
  const uint32_t codes = *reinterpret_cast<const uint32_t*>(packed + row * (K / 2) + k0 / 2);
  const float scale = e4m3_to_f32(sb[row * (K / 16) + k0 / 16]);
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t byte = codes >> (8 * i);
    const __nv_bfloat162 h = __floats2bfloat162_rn(e2m1_to_f32(byte & 0xF) * scale,
                                                   e2m1_to_f32((byte >> 4) & 0xF) * scale);
    o[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  const long long row_bytes = K * 2;
  const long long rb = row >> 7, r = row & 127, kb = (k0 * 2) >> 7, ch = ((k0 * 2) & 127) >> 4;
  const long long dst_off =
      (((rb * (row_bytes / 128)) + kb) * 128 + r) * 128 + ((ch ^ (r & 7)) * 16);
  *reinterpret_cast<uint4*>(dst + dst_off) = make_uint4(o[0], o[1], o[2], o[3]);
}

__global__ void __launch_bounds__(256)
    sf_relayout_kernel(const uint8_t* src, uint8_t* dst, long long rows, long long nsc) {
  const long long na = nsc / 4;  // 512-byte tiles per 128-row block
  const long long q = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
  if (q >= rows * na) return;
  const long long row = q / na, a = q - row * na;
  const uint32_t word = *reinterpret_cast<const uint32_t*>(src + row * nsc + 4 * a);
  const long long rb = row >> 7, r = row & 127;
  *reinterpret_cast<uint32_t*>(dst + (rb * na + a) * 512 + (r & 31) * 16 + 4 * (r >> 5)) = word;
}

__global__ void __launch_bounds__(256)
    fill_expert_scale_kernel(const float* g, float* dst, int E, long long per) {
  const long long i = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
  if (i < E * per) dst[i] = g[i / per];
}

template <typename Kern, typename Param>
cudaError_t launch_simple(Kern k, dim3 grid, dim3 block, const Param& prm, cudaStream_t s,
                          bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, prm);
}

}  // namespace

cudaError_t launch_route(const RouteParams& p, cudaStream_t s, bool pdl) {
  const long long warps =
      static_cast<long long>(p.M) * ((p.L / 128 + ROUTE_QG - 1) / ROUTE_QG + 1);
  const int blocks = static_cast<int>((warps + ROUTE_WARPS - 1) / ROUTE_WARPS);
  return launch_simple(route_quant_kernel, dim3(blocks), dim3(32 * ROUTE_WARPS), p, s, pdl);
}
cudaError_t launch_perm_hist(const PermParams& p, cudaStream_t s, bool pdl) {
  return launch_simple(perm_hist_kernel, dim3(p.nblocks), dim3(PERM_BLOCK), p, s, pdl);
}
cudaError_t launch_perm_scatter(const PermParams& p, cudaStream_t s, bool pdl) {
  return launch_simple(perm_scatter_kernel, dim3(p.nblocks), dim3(PERM_BLOCK), p, s, pdl);
}
cudaError_t launch_perm_gather(const PermParams& p, cudaStream_t s, bool pdl) {
  long long chunks = static_cast<long long>(p.M) * p.k * (p.zrow / 16);
  if (chunks < static_cast<long long>(p.M) * p.k * (p.L / 128))  // zsT transposition
    chunks = static_cast<long long>(p.M) * p.k * (p.L / 128);
  if (p.zsf_t != nullptr) {
    const long long sf = static_cast<long long>(p.sf_tiles) * 128 * (p.L / p.sf_group / 4);
    chunks = chunks > sf ? chunks : sf;
  }
  return launch_simple(perm_gather_kernel, dim3(static_cast<unsigned>((chunks + 255) / 256)),
                       dim3(256), p, s, pdl);
}
cudaError_t launch_route_small(const RouteParams& rp, const PermParams& p, cudaStream_t s,
                               bool pdl) {
  const long long items =
      static_cast<long long>(rp.M) * rp.k * ((rp.L / 128 + ROUTE_QG - 1) / ROUTE_QG);
  constexpr int NW = SMALL_THREADS / 32;
  const int blocks = static_cast<int>((items + NW - 1) / NW);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(SMALL_THREADS);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, route_small_kernel, rp, p);
}
cudaError_t launch_norm(const NormParams& p, cudaStream_t s, bool pdl) {
  return launch_simple(norm_kernel, dim3(p.M), dim3(128), p, s, pdl);
}

cudaError_t launch_nvfp4_expand(const uint8_t* packed, const uint8_t* sb, void* dst,
                                long long rows, long long K, cudaStream_t s) {
  const long long chunks = rows * (K / 8);
  nvfp4_expand_kernel<<<static_cast<unsigned>((chunks + 255) / 256), 256, 0, s>>>(
      packed, sb, static_cast<uint8_t*>(dst), rows, K);
  return cudaGetLastError();
}
cudaError_t launch_fill_expert_scale(const float* g, float* dst, int E, long long per,
                                     cudaStream_t s) {
  const long long n = E * per;
  fill_expert_scale_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(g, dst, E,
                                                                                    per);
  return cudaGetLastError();
}
cudaError_t launch_sf_relayout(const uint8_t* src, uint8_t* dst, long long rows, long long nsc,
                               cudaStream_t s) {
  const long long n = rows * (nsc / 4);
  sf_relayout_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(src, dst, rows,
                                                                              nsc);
  return cudaGetLastError();
}
cudaError_t launch_tile_relayout(const void* src, void* dst, long long rows, long long row_bytes,
                                 cudaStream_t s) {
  const long long chunks = rows * (row_bytes / 16);
  tile_relayout_kernel<<<static_cast<unsigned>((chunks + 255) / 256), 256, 0, s>>>(
      static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), rows, row_bytes);
  return cudaGetLastError();
}

}  // namespace klt
