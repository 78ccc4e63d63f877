// train_attn_bwd.cu - mars_train_attn_bwd: dQ, dK, dV of the MARS masked
// attention over z = [x ; x~].
//
// Method: "MARS: Enabling Autoregressive Models Multi-Token Generation",
// Sec. 3.2 (Eq. 1, Eq. 2: both streams share one forward, so one backward
// carries the gradients of the losses of Eqs. 3 and 5 to q, k and v).  For one
// head, with S = scale q k^T, P = softmax(S + M) and O = P v:
//   dV = P^T dO,  dP = dO v^T,  dS = P * (dP - delta),  delta_i = sum_d dO_i O_i,
//   dQ = scale dS k,  dK = scale dS^T q,
// and P is recomputed from the forward's log-sum-exp: P = exp(S - lse).
//
// sm_103a design (tensor-bound).  Four launches, deterministic (the only atomic
// hands out work units):
//   1. delta_kernel: delta_i = rowsum(dO_i * O_i), fp32, 16-byte loads.
//   2. bwd_kernel<kDKV>: one unit per (sequence, KV head, 128-key tile, chunk of
//      the group's query heads).  For every query head of the chunk and every
//      128-row query tile that sees the key tile (an exact interval test on
//      Eq. 2's structure) tcgen05 computes dP = dO V^T and S = Q K^T into
//      tensor memory; the elementwise warps form P and dS and write them to
//      shared memory as SW128 [128 rows x 64 keys] tiles; tcgen05 then
//      accumulates dV += P^T dO and dK += dS^T Q in tensor memory (P / dS read
//      MN-major as the A operand, Q / dO MN-major as B) over the whole chunk.
//      A group is split into chunks only on the heavy key tiles (so that no unit
//      serialises a large share of the work on one SM); a one-chunk unit writes
//      bf16 dK, dV directly, a split one an fp32 partial per chunk.
//   3. reduce_kernel (GQA): the chunks' partials of the split tiles, summed in
//      chunk order.
//   4. bwd_kernel<kDQ>: one unit per (sequence, query head, 128-row query tile):
//      the same dP, S, dS for every key tile the query tile sees, then
//      dQ += dS K (dS K-major, K MN-major).
// CTAs are persistent (one per SM) and take units heaviest first from a work
// counter.  Roles: warp 0 TMA producer (the unit's fixed tiles, then a ring of
// single-tile slots with the per-step tiles, each slot freed by the commit after
// its last reader), warp 1 MMA issuer (one elected lane), warps 2..5 and 6..9
// elementwise (thread = TMEM lane = query row; warpgroup e takes keys
// [64 e, 64 e + 64): P and dS need only per-row constants, so the halves
// exchange nothing).  The elementwise warps release S, dP as soon as they hold
// them in registers, so the next step's products overlap their work.  Every
// mbarrier wait is bounded; a wait that gives up sets MARS_DEV_TIMEOUT.
#include <cuda.h>

#include <algorithm>
#include <climits>
#include <functional>
#include <mutex>
#include <queue>
#include <vector>

#include "common.cuh"

namespace {

using namespace mars;

constexpr int kT = 128;            // query rows of a query tile = keys of a key tile
constexpr int kBox = 128 * 128;    // bytes of one [128 rows x 64 bf16] SW128 box
constexpr int kEW = 2;             // elementwise warpgroups, each 128 / kEW keys of a step
constexpr int kEWCols = kT / kEW;
static_assert(kEWCols % 32 == 0, "the visibility mask is built per 32 columns");
constexpr int kThreads = 64 + 128 * kEW;  // producer, MMA issuer, elementwise warps
constexpr int kMaxTiles = 1024;    // tiles per batch entry and head (2 * ceil(L / 128))

enum Mode { kDKV = 0, kDQ = 1 };
// (d0, d1) = (dp0 - t, dp1 - t) * (p0, p1) with packed fp32x2 arithmetic.
__device__ __forceinline__ void sub_mul2(float dp0, float dp1, float t, float p0, float p1, float& d0, float& d1) {
  asm("{\n .reg .b64 x, c, p, r;\n mov.b64 x, {%2, %3};\n mov.b64 c, {%4, %4};\n mov.b64 p, {%5, %6};\n"
      " sub.rn.f32x2 r, x, c;\n mul.rn.f32x2 r, r, p;\n mov.b64 {%0, %1}, r;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(dp0), "f"(dp1), "f"(t), "f"(p0), "f"(p1));
}

template <int D, int MODE>
struct BCfg {
  static constexpr int NB = D / 64;
  static constexpr int TILE = NB * kBox;  // one [128 x D] bf16 tile
  // dKV: the unit's K and V once; one ring of single-tile slots takes dO(n), Q(n),
  // dO(n + 1), ... in that order.  dQ: the unit's Q and dO once; K and V in two
  // rings (3 K slots, loaded first, so K(n + 1) waits only for dQ(n - 2); V(n) is
  // read by dP(n) alone and frees its slot early).  Both: P (dKV only) and dS
  // [128 x 128] tiles.  A slot is released by the commit after the last product
  // that reads it, so the next steps' tiles load while this step's products run.
  static constexpr bool SPLIT = MODE == kDQ;
  static constexpr int NX = SPLIT ? (D == 128 ? 1 : 2) : 0, NY = SPLIT ? 3 : 0;  // V, K slots (dQ)
  static constexpr int NSLOT = SPLIT ? NX + NY : (D == 128 ? 3 : 6);  // 3: 225 KB of 227 at D = 128
  // S(n + 1) ahead of step n's accumulating products needs its tile while step n's
  // are still held: at least four slots in the single ring; always with two rings.
  // With three, only dP(n + 1) goes ahead.
  static constexpr bool EARLY_S = SPLIT || NSLOT >= 4;
  static constexpr int FIXED_OFF = 0;                   // K, V (dKV) or Q, dO (dQ)
  static constexpr int RING_OFF = FIXED_OFF + 2 * TILE;
  static constexpr int P_OFF = RING_OFF + NSLOT * TILE;
  static constexpr int DS_OFF = P_OFF + (MODE == kDKV ? 2 * kBox : 0);
  static constexpr int SMEM = DS_OFF + 2 * kBox + 1024;  // + slack to align the base to 1024
  static constexpr int S_COL = 0, DP_COL = kT, ACC_COL = 2 * kT;  // ACC: dK | dV, or dQ
  static_assert(SMEM <= 232448, "shared memory");
  static_assert(ACC_COL + (MODE == kDKV ? 2 : 1) * D <= 512, "tensor memory");
};

// Work units, heaviest first.  An entry is (tile, chunk, chunks): bits 0..15 the
// tile (0 .. 2 nt - 1), 16..23 the chunk, 24..31 the number of chunks its GQA group
// is split into.  dKV: entry x (batch, KV head) units, each summing dK, dV over the
// chunk's query heads (one chunk: the whole group, written as bf16 directly; more:
// an fp32 partial per chunk, summed by reduce_kernel).  dQ: entry x (batch, query
// head) units, one chunk each.
// The order is a kernel parameter, copied with every launch, so a small one (3 KB)
// is used when the entries and tiles fit (each KB of parameter delays the launch).
constexpr int kMaxEntries = 4096;
constexpr int kSmallEntries = 512, kSmallTiles = 128;
template <int NE, int NT>
struct UnitOrderT {
  uint32_t entry[NE];
  // per tile: its steps' other tiles, [lo0, hi0) in the clean stream and [lo1, hi1)
  // in the noisy one (the same for every unit of the tile)
  uint16_t rng[NT][4];
  int n;
};
using UnitOrder = UnitOrderT<kMaxEntries, kMaxTiles>;
using SmallOrder = UnitOrderT<kSmallEntries, kSmallTiles>;
// Chunks per tile (dKV), for reduce_kernel: tiles with one chunk are already final.
struct ChunkTable {
  uint8_t nch[kMaxTiles];
};

struct BwdArgs {
  const float* lse;    // [b, Hq, 2L] natural log
  const float* delta;  // [b, Hq, 2L]
  float* part;         // GQA: per-query-head fp32 dK | dV partials [2][b, 2L, Hq, D]; nullptr when G == 1
  int* next_unit;      // work counter of the launch (zeroed by delta_kernel)
  uint16_t* dq;
  uint16_t* dk;
  uint16_t* dv;
  int32_t* status;
  int batch, L, B, Hq, Hkv, G;
  int nt;              // tiles per stream: ceil(L / 128)
  float scale_log2;    // scale * log2(e)
  float scale;
};

// Tile t of the 2 * nt tiles of z: stream t / nt, rows [r0, r0 + 128) cut at end.
__host__ __device__ __forceinline__ void tile_rows(const BwdArgs& a, int t, int& r0, int& end) {
  const bool noisy = t >= a.nt;
  const int j = noisy ? t - a.nt : t;
  r0 = (noisy ? a.L : 0) + kT * j;
  end = noisy ? 2 * a.L : a.L;
}

// Does any query row of query tile qt see any key of key tile kt (Eq. 2)?
__host__ __device__ __forceinline__ bool tile_visible(const BwdArgs& a, int qt, int kt) {
  int q0, qe, k0, ke;
  tile_rows(a, qt, q0, qe);
  tile_rows(a, kt, k0, ke);
  const int q1 = min(q0 + kT, qe) - 1, k1 = min(k0 + kT, ke) - 1;
  if (q0 < a.L) return k0 < a.L && q1 >= k0;  // clean rows see the clean causal prefix
  // noisy rows t = i - L see clean [0, B * (t / B) - 1] and noisy [L + B * (t / B), i]
  if (k0 < a.L) return a.B * ((q1 - a.L) / a.B) - 1 >= k0;
  const int i = max(q0, k0);
  return i <= q1 && a.L + a.B * ((i - a.L) / a.B) <= k1;
}

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;  // descriptor version for sm_100-class tensor cores
  d |= 2ull << 61;  // 128-byte swizzle
  return d;
}

// bf16 x bf16 -> fp32, M x N; a_mn / b_mn: the operand is MN-major (transposed).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------- delta
// delta_i = sum_d dO_i O_i in fp32.  A row of D bf16 is D / 8 threads, each
// reading one 16-byte chunk of O and of dO; the chunk sums meet by shuffles
// inside the row's lanes (D / 8 divides 32).
__global__ void __launch_bounds__(256) delta_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                                                    float* __restrict__ delta, int* __restrict__ counters, int batch,
                                                    int n2, int Hq, int D) {
  // launched as a programmatic dependent: nothing global is touched before the
  // previous kernel in the stream has completed; the next kernel may start its set-up
  griddep_wait();
  griddep_launch_dependents();
  if (blockIdx.x == 0 && threadIdx.x < 2) counters[threadIdx.x] = 0;  // the two work counters of bwd_kernel
  const int per_row = D / 8;
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long row = tid / per_row;  // (b, i, h)
  const int c = static_cast<int>(tid % per_row);
  const bool valid = row < static_cast<long long>(batch) * n2 * Hq;
  float acc = 0.f;
  if (valid) {
    const uint4 wo = __ldg(reinterpret_cast<const uint4*>(o + row * D) + c);
    const uint4 wd = __ldg(reinterpret_cast<const uint4*>(dout + row * D) + c);
    const uint32_t po[4] = {wo.x, wo.y, wo.z, wo.w}, pd[4] = {wd.x, wd.y, wd.z, wd.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(bf16lo_to_f32(po[e]), bf16lo_to_f32(pd[e]), acc);
      acc = fmaf(bf16hi_to_f32(po[e]), bf16hi_to_f32(pd[e]), acc);
    }
  }
  for (int s = per_row / 2; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (valid && c == 0) {
    const int h = static_cast<int>(row % Hq);
    const long long bi = row / Hq;
    const int i = static_cast<int>(bi % n2), b = static_cast<int>(bi / n2);
    delta[(static_cast<size_t>(b) * Hq + h) * n2 + i] = acc;
  }
}

// ---------------------------------------------------------------- GQA reduction
// dK (m = 0) and dV (m = 1) of KV head g on the key tiles whose GQA group was split
// into chunks: the sum of the chunks' fp32 partials (slots g G + c), in chunk order,
// rounded once to bf16.  Tiles of one chunk were written by the dK/dV pass.  Thread =
// 8 consecutive elements.
__global__ void __launch_bounds__(256) reduce_kernel(const float* __restrict__ part, uint16_t* __restrict__ dk,
                                                     uint16_t* __restrict__ dv, int batch, int L, int nt, int Hkv,
                                                     int G, int D, const __grid_constant__ ChunkTable ct) {
  griddep_wait();  // programmatic dependent launch, as delta_kernel
  griddep_launch_dependents();
  const int n2 = 2 * L;
  const long long e8 = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long per_m = static_cast<long long>(batch) * n2 * Hkv * D / 8;
  if (e8 >= 2 * per_m) return;
  const int m = static_cast<int>(e8 / per_m);
  const long long r = e8 % per_m;
  const int dc = static_cast<int>(r % (D / 8));
  const long long rg = r / (D / 8);  // (b, i, g)
  const int g = static_cast<int>(rg % Hkv);
  const long long bi = rg / Hkv;
  const int i = static_cast<int>(bi % n2);
  const int nch = ct.nch[i < L ? i / kT : nt + (i - L) / kT];
  if (nch <= 1) return;  // final already
  const int Hq = Hkv * G;
  const float* src = part + ((static_cast<size_t>(m) * batch * n2 + bi) * Hq + static_cast<size_t>(g) * G) * D + 8 * dc;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int h = 0; h < nch; ++h) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(src + static_cast<size_t>(h) * D));
    const float4 y = __ldg(reinterpret_cast<const float4*>(src + static_cast<size_t>(h) * D + 4));
    acc[0] += x.x; acc[1] += x.y; acc[2] += x.z; acc[3] += x.w;
    acc[4] += y.x; acc[5] += y.y; acc[6] += y.z; acc[7] += y.w;
  }
  uint16_t* dst = (m == 0 ? dk : dv) + (rg * D + 8 * dc);
  *reinterpret_cast<uint4*>(dst) = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                              pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
}

// ---------------------------------------------------------------- main kernel
template <int D, int MODE, int NE, int NT>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do, const BwdArgs a,
               const __grid_constant__ UnitOrderT<NE, NT> order) {
  using C = BCfg<D, MODE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar_fixed, bar_ffree, bar_stage[C::NSLOT], bar_free[C::NSLOT], bar_s, bar_sdp, bar_p, bar_pfree,
      bar_acc, bar_stg;
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- units: (b, query head, key tile) for dKV, (b, query head, query tile) for
  // dQ, listed heaviest tile first.  The CTAs are persistent: each takes its first
  // unit by its index and every further one from the launch's work counter, so
  // the heavy units spread over the SMs and the light ones fill in behind them.
  // The producer fetches; it publishes the r-th unit of the CTA in queue slot
  // r % 4 (bar_unit[r % 4]) for the other roles.  It runs at most three units
  // ahead of the elementwise warps (it fetches unit r + 2 only after unit r's last
  // S, which comes after the elementwise warps' P of unit r - 1), so four slots
  // suffice.
  const int per_entry = MODE == kDKV ? a.batch * a.Hkv : a.batch * a.Hq;
  const int nunits = order.n * per_entry;
  // A unit's steps: every query tile that sees its key tile (dKV), or every key tile
  // its query tile sees (dQ), in index order.  The conditions of Eq. 2 are monotonic
  // in the other tile's index within a stream, so those tiles form one range per
  // stream, [lo0, hi0) among the clean tiles and [lo1, hi1) among the noisy ones.
  // The host finds the ranges once per tile; the producer publishes them with the unit.
  struct Unit {
    int tile, b, hh, g, chunk, nch, h_lo, h_hi, u0, uend, nsteps, lo0, hi0, lo1, hi1;
  };
  __shared__ int unit_q[4];
  __shared__ int4 unit_rng[4];
  __shared__ __align__(8) uint64_t bar_unit[4];
  auto unit_base = [&](int u, Unit& U) {
    const uint32_t e = order.entry[u / per_entry];
    const int rest = u % per_entry;
    U.tile = static_cast<int>(e & 0xFFFFu);
    U.chunk = static_cast<int>((e >> 16) & 0xFFu);
    U.nch = static_cast<int>(e >> 24);
    if (MODE == kDKV) {  // query heads [h_lo, h_hi) of KV head g's group
      U.b = rest / a.Hkv;
      U.g = rest % a.Hkv;
      U.h_lo = U.g * a.G + (U.chunk * a.G) / U.nch;
      U.h_hi = U.g * a.G + ((U.chunk + 1) * a.G) / U.nch;
      U.hh = U.h_lo;
    } else {  // one query head
      U.b = rest / a.Hq;
      U.hh = rest % a.Hq;
      U.g = U.hh / a.G;
      U.h_lo = U.hh;
      U.h_hi = U.hh + 1;
    }
    tile_rows(a, U.tile, U.u0, U.uend);
  };
  auto set_ranges = [&](Unit& U, int lo0, int hi0, int lo1, int hi1) {
    U.lo0 = lo0, U.hi0 = hi0, U.lo1 = lo1, U.hi1 = hi1;
    U.nsteps = (U.h_hi - U.h_lo) * ((hi0 - lo0) + (hi1 - lo1));  // (head, other tile) pairs
  };
  // the r-th unit of this CTA as the consumers see it: false at the end (or on a timeout)
  auto unit = [&](int r, Unit& U) -> bool {
    if (!mbar_wait(&bar_unit[r & 3], (r >> 2) & 1)) {
      set_status(a.status, MARS_DEV_TIMEOUT);
      return false;
    }
    const int u = unit_q[r & 3];
    if (u < 0) return false;
    unit_base(u, U);
    const int4 rg = unit_rng[r & 3];
    set_ranges(U, rg.x, rg.y, rg.z, rg.w);
    return true;
  };
  // the unit's first step tile after o (o = -1: its first)
  auto next_other = [&](const Unit& U, int o) {
    ++o;
    if (o < U.lo0) o = U.lo0;
    if (o >= U.hi0 && o < U.lo1) o = U.lo1;
    return o;
  };
  // the unit's next step (query head h, other tile o), heads outermost; h < 0 before
  // the first step
  auto next_step = [&](const Unit& U, int& h, int& o) {
    if (h < 0) {
      h = U.h_lo;
      o = next_other(U, -1);
      return;
    }
    o = next_other(U, o);
    if (o >= U.hi1) {
      ++h;
      o = next_other(U, -1);
    }
  };

  if (threadIdx.x == 0) {
    mbar_init(&bar_fixed, 1);
    mbar_init(&bar_ffree, 1);  // a unit's last S and dP have read the fixed tiles
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(&bar_stage[s], 1);
      mbar_init(&bar_free[s], 1);
    }
    mbar_init(&bar_s, 1);
    mbar_init(&bar_sdp, 128 * kEW);  // S(n), dP(n) are in the elementwise warps' registers
    mbar_init(&bar_p, 128 * kEW);
    mbar_init(&bar_pfree, 1);  // step n's accumulating products are complete
    mbar_init(&bar_acc, 1);
    mbar_init(&bar_stg, 128 * kEW);  // every elementwise warp has written its staged epilogue block out
    for (int s = 0; s < 4; ++s) mbar_init(&bar_unit[s], 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  // Programmatic dependent launch: the set-up above overlaps the previous kernel.
  // The dK/dV pass touches nothing global before that kernel has completed.  The dQ
  // pass reads only what delta_kernel and the caller wrote: it starts once the
  // kernel before it (the GQA reduction, or the dK/dV pass) has released its
  // dependents, which each does after its own wait, so those writes are complete;
  // the dQ pass waits at its end instead, so it runs beside the reduction and still
  // completes after it.
  if constexpr (MODE == kDKV) griddep_wait();
  const uint32_t fixed_s = smem_u32(smem + C::FIXED_OFF);
  const uint32_t ring_s = smem_u32(smem + C::RING_OFF);
  const uint32_t p_s = smem_u32(smem + C::P_OFF);
  const uint32_t ds_s = smem_u32(smem + C::DS_OFF);
  bool ok = true;
  // Ring slot of step g's tile y (0: dO or V, 1: Q or K) and which fill of that
  // slot it is (the parity of its barriers).
  auto slot_of = [&](int g, int y, int& sl, int& k) {
    if constexpr (C::SPLIT) {
      sl = y == 0 ? g % C::NX : C::NX + g % C::NY;
      k = y == 0 ? g / C::NX : g / C::NY;
    } else {
      const int tt = 2 * g + y;
      sl = tt % C::NSLOT;
      k = tt / C::NSLOT;
    }
  };

  if (warp == 0) {
    // ================= TMA producer
    if (lane == 0) {
      int gp = 0;  // steps whose tiles were issued (over all units)
      Unit U;
      for (int r = 0; ok; ++r) {
        const int u = r == 0 ? static_cast<int>(blockIdx.x) : static_cast<int>(gridDim.x) + atomicAdd(a.next_unit, 1);
        if (u < nunits) {
          unit_base(u, U);
          const uint16_t* rg = order.rng[U.tile];
          set_ranges(U, rg[0], rg[1], rg[2], rg[3]);
          unit_rng[r & 3] = make_int4(U.lo0, U.hi0, U.lo1, U.hi1);
          // the unit's fixed tiles toward L2 now: they load once the previous unit's
          // last S and dP have read the current ones
          for (int c = 0; c < C::NB; ++c) {
            if (MODE == kDKV) {
              tma_prefetch_l2_4d(&tm_k, 64 * c, U.g, U.u0, U.b);
              tma_prefetch_l2_4d(&tm_v, 64 * c, U.g, U.u0, U.b);
            } else {
              tma_prefetch_l2_4d(&tm_q, 64 * c, U.hh, U.u0, U.b);
              tma_prefetch_l2_4d(&tm_do, 64 * c, U.hh, U.u0, U.b);
            }
          }
        }
        unit_q[r & 3] = u < nunits ? u : -1;
        mbar_arrive(&bar_unit[r & 3]);  // release: the slot is written
        if (u >= nunits) break;
        // fixed operands: K, V of the key tile (dKV) or Q, dO of the query tile (dQ),
        // once the previous unit's last S and dP have read theirs
        if (r > 0 && !mbar_wait(&bar_ffree, (r - 1) & 1)) {
          set_status(a.status, MARS_DEV_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(&bar_fixed, 2 * C::TILE);
        for (int c = 0; c < C::NB; ++c) {
          if (MODE == kDKV) {
            tma_load_4d(fixed_s + c * kBox, &tm_k, &bar_fixed, 64 * c, U.g, U.u0, U.b);
            tma_load_4d(fixed_s + C::TILE + c * kBox, &tm_v, &bar_fixed, 64 * c, U.g, U.u0, U.b);
          } else {
            tma_load_4d(fixed_s + c * kBox, &tm_q, &bar_fixed, 64 * c, U.hh, U.u0, U.b);
            tma_load_4d(fixed_s + C::TILE + c * kBox, &tm_do, &bar_fixed, 64 * c, U.hh, U.u0, U.b);
          }
        }
        for (int n = 0, hs = -1, ot = -1; ok && n < U.nsteps; ++n) {
          next_step(U, hs, ot);
          int o0, oe;
          tile_rows(a, ot, o0, oe);
          for (int j = 0; j < 2; ++j) {  // ring tiles of a step: dO, Q (dKV) or K, V (dQ)
            const int y = C::SPLIT ? 1 - j : j;
            int sl, k;
            slot_of(gp, y, sl, k);
            if (k > 0 && !mbar_wait(&bar_free[sl], (k - 1) & 1)) {
              set_status(a.status, MARS_DEV_TIMEOUT);
              ok = false;
              break;
            }
            const CUtensorMap* tm = MODE == kDKV ? (y ? &tm_q : &tm_do) : (y ? &tm_k : &tm_v);
            const int hc = MODE == kDKV ? hs : U.g;
            const uint32_t dst = ring_s + sl * C::TILE;
            mbar_arrive_expect_tx(&bar_stage[sl], C::TILE);
            for (int c = 0; c < C::NB; ++c) tma_load_4d(dst + c * kBox, tm, &bar_stage[sl], 64 * c, hc, o0, U.b);
          }
          ++gp;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer (whole warp runs the schedule, one elected lane issues)
    const bool leader = elect_one();
    constexpr uint32_t id_s = idesc_bf16(kT, kT, false, false);   // S, dP: A, B K-major
    constexpr uint32_t id_acc = MODE == kDKV ? idesc_bf16(kT, D, true, true)   // P^T dO, dS^T Q
                                             : idesc_bf16(kT, D, false, true); // dS K
    auto wait_all = [&](uint64_t* bar, int parity) { ok = ok && __all_sync(0xffffffffu, mbar_wait(bar, parity)); };
    // Ring tiles of step n: x = 2n (dO or V) and y = 2n + 1 (Q or K); the fixed
    // tiles are the others.
    auto tiles = [&](int n, uint32_t& q_t, uint32_t& do_t, uint32_t& k_t, uint32_t& v_t) {
      int sx, sy, kx, ky;
      slot_of(n, 0, sx, kx);
      slot_of(n, 1, sy, ky);
      const uint32_t x_t = ring_s + sx * C::TILE, y_t = ring_s + sy * C::TILE;
      q_t = MODE == kDKV ? y_t : fixed_s;
      do_t = MODE == kDKV ? x_t : fixed_s + C::TILE;
      k_t = MODE == kDKV ? fixed_s : y_t;
      v_t = MODE == kDKV ? fixed_s + C::TILE : x_t;
    };
    // dP(n) = dO V^T (its ring tile x is loaded first)
    auto issue_dp = [&](int n) {
      int sx, kx;
      slot_of(n, 0, sx, kx);
      wait_all(&bar_stage[sx], kx & 1);
      if (!ok) return;
      tc_fence_after();
      uint32_t q_t, do_t, k_t, v_t;
      tiles(n, q_t, do_t, k_t, v_t);
      if (leader) {
        const uint64_t ddo = smem_desc(do_t, 16, 1024), dv_ = smem_desc(v_t, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = ((ks >> 2) * kBox + (ks & 3) * 32) >> 4;
          tc_mma_ss(tmem + C::DP_COL, ddo + off, dv_ + off, id_s, ks > 0 ? 1u : 0u);
        }
        if (MODE == kDQ) tc_commit(&bar_free[sx]);  // V(n) has no other reader
      }
      __syncwarp();
    };
    // S(n) = Q K^T, then "S(n) and dP(n) ready" (and, after a unit's last step,
    // "the fixed tiles may be replaced")
    auto issue_s = [&](int n, bool unit_last) {
      int sy, ky;
      slot_of(n, 1, sy, ky);
      wait_all(&bar_stage[sy], ky & 1);
      if (!ok) return;
      tc_fence_after();
      uint32_t q_t, do_t, k_t, v_t;
      tiles(n, q_t, do_t, k_t, v_t);
      if (leader) {
        const uint64_t dq_ = smem_desc(q_t, 16, 1024), dk_ = smem_desc(k_t, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = ((ks >> 2) * kBox + (ks & 3) * 32) >> 4;
          tc_mma_ss(tmem + C::S_COL, dq_ + off, dk_ + off, id_s, ks > 0 ? 1u : 0u);
        }
        tc_commit(&bar_s);
        if (unit_last) tc_commit(&bar_ffree);
      }
      __syncwarp();
    };
    // the accumulating products of step n, once its P and dS are in shared memory;
    // the first step of a unit starts the accumulators afresh
    auto issue_acc = [&](int n, bool first, bool last) {
      wait_all(&bar_p, n & 1);
      if (!ok) return;
      tc_fence_after();
      int sx, sy, kx, ky;
      slot_of(n, 0, sx, kx);
      slot_of(n, 1, sy, ky);
      uint32_t q_t, do_t, k_t, v_t;
      tiles(n, q_t, do_t, k_t, v_t);
      if (leader) {
        if (MODE == kDKV) {
          // dV += P^T dO and dK += dS^T Q over the 128 query rows (16 per step)
          const uint64_t dpa = smem_desc(p_s, kBox, 1024), dsa = smem_desc(ds_s, kBox, 1024);
          const uint64_t ddo = smem_desc(do_t, kBox, 1024), dqb = smem_desc(q_t, kBox, 1024);
#pragma unroll
          for (int ks = 0; ks < kT / 16; ++ks) {
            const uint32_t off = (ks * 16 * 128) >> 4;
            tc_mma_ss(tmem + C::ACC_COL + D, dpa + off, ddo + off, id_acc, (!first || ks > 0) ? 1u : 0u);
          }
          tc_commit(&bar_free[sx]);  // dO(n): read by dP and dV, both issued
#pragma unroll
          for (int ks = 0; ks < kT / 16; ++ks) {
            const uint32_t off = (ks * 16 * 128) >> 4;
            tc_mma_ss(tmem + C::ACC_COL, dsa + off, dqb + off, id_acc, (!first || ks > 0) ? 1u : 0u);
          }
        } else {
          // dQ += dS K over the 128 keys (16 per step): dS K-major, K MN-major
          const uint64_t dsa = smem_desc(ds_s, 16, 1024), dkb = smem_desc(k_t, kBox, 1024);
#pragma unroll
          for (int ks = 0; ks < kT / 16; ++ks) {
            const uint32_t aoff = ((ks >> 2) * kBox + (ks & 3) * 32) >> 4, boff = (ks * 16 * 128) >> 4;
            tc_mma_ss(tmem + C::ACC_COL, dsa + aoff, dkb + boff, id_acc, (!first || ks > 0) ? 1u : 0u);
          }
        }
        tc_commit(&bar_free[sy]);  // Q(n) (read by S, dK) or K(n) (read by S, dQ)
        tc_commit(&bar_pfree);     // the P / dS tiles may be overwritten
        if (last) tc_commit(&bar_acc);
      }
      __syncwarp();
    };
    // Step n + 1's dP (and S, when the ring holds both of its tiles beside step
    // n's) is issued as soon as the elementwise warps hold S(n), dP(n) in
    // registers, so the tensor cores work while P(n), dS(n) are formed.  Steps are
    // numbered over all the units of the CTA (gs); a unit's first dP and S may run
    // while the elementwise warps write the previous unit's accumulators out.
    int gs = 0;
    Unit U;
    for (int r = 0; ok && unit(r, U); ++r) {
      wait_all(&bar_fixed, r & 1);
      if (!ok) break;
      tc_fence_after();
      const int N = U.nsteps;
      if (N == 0) {
        if (leader) tc_commit(&bar_ffree);
        __syncwarp();
        continue;
      }
      issue_dp(gs);
      issue_s(gs, N == 1);
      for (int n = 0; ok && n < N; ++n, ++gs) {
        const bool next = n + 1 < N;
        if (next) {
          wait_all(&bar_sdp, gs & 1);
          issue_dp(gs + 1);
          if (C::EARLY_S) issue_s(gs + 1, n + 2 == N);
        }
        issue_acc(gs, n == 0, n + 1 == N);
        if (next && !C::EARLY_S) issue_s(gs + 1, n + 2 == N);
      }
    }
    if (!ok && leader) set_status(a.status, MARS_DEV_TIMEOUT);
    __syncwarp();
  } else {
    // ================= elementwise: thread = TMEM lane = row of S (a query row)
    const int ew = (warp - 2) >> 2;  // warpgroup: keys [kEWCols ew, kEWCols (ew + 1)) of the tile
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    int gs = 0, nacc = 0;  // steps done (over all units), units whose accumulators were read
    int nstg = 0;          // epilogue blocks written out (phases of bar_stg)
    Unit U;
    for (int ur = 0; ok && unit(ur, U); ++ur) {
      const int b = U.b, hh = U.hh, g = U.g, tile = U.tile, u0 = U.u0, uend = U.uend, nsteps = U.nsteps;
      for (int n = 0, hs = -1, ot = -1; n < nsteps; ++n, ++gs) {
        next_step(U, hs, ot);
        const int head = hs;
        // query tile and key tile of this step
        const int qt = MODE == kDKV ? ot : tile, kt = MODE == kDKV ? tile : ot;
        int q0, qe, k0, ke;
        tile_rows(a, qt, q0, qe);
        tile_rows(a, kt, k0, ke);
        const int i = q0 + r;
        const bool row_ok = i < qe;
        // visible keys of row i (Eq. 2): clean [0, c_hi], noisy [n_lo, n_hi]
        int c_hi = -1, n_lo = 1, n_hi = 0;
        if (row_ok) {
          if (i < a.L) {
            c_hi = i;
          } else {
            const int c = a.B * ((i - a.L) / a.B);
            c_hi = c - 1;
            n_lo = a.L + c;
            n_hi = i;
          }
        }
        const size_t ri = (static_cast<size_t>(b) * a.Hq + head) * (2 * a.L) + (row_ok ? i : 0);
        const float lse2 = row_ok ? __ldg(a.lse + ri) * kLog2e : 0.f;
        const float dlt = row_ok ? __ldg(a.delta + ri) : 0.f;
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_s, gs & 1));
        if (!ok) break;
        tc_fence_after();
        {
          // keys [c0, c0 + kEWCols) of the tile: chunks [qb, qb + kEWCols / 8) of SW128 box hb
          const int c0 = kEWCols * ew, hb = c0 / 64, qb = (c0 % 64) / 8;
          constexpr int NC = kEWCols / 8;  // 16-byte chunks per row
          uint32_t sv[kEWCols], dpv[kEWCols];
#pragma unroll
          for (int c = 0; c < kEWCols; c += 32) {
            tmem_ld32(tmem + lane_addr + C::S_COL + c0 + c, *reinterpret_cast<uint32_t(*)[32]>(&sv[c]));
            tmem_ld32(tmem + lane_addr + C::DP_COL + c0 + c, *reinterpret_cast<uint32_t(*)[32]>(&dpv[c]));
          }
          // The row's visible keys in this slice as local columns [vlo, vhi] (empty when
          // vlo > vhi): a key tile lies in one stream, so one interval of Eq. 2 applies.
          const int kb = k0 + c0;
          const bool clean_keys = k0 < a.L;
          const int vlo = (clean_keys ? 0 : n_lo) - kb;
          const int vhi = min(clean_keys ? c_hi : n_hi, ke - 1) - kb;
          const bool full = __all_sync(0xffffffffu, vlo <= 0 && vhi >= kEWCols - 1);  // interior: no mask
          tc_wait_ld();
          tc_fence_before();
          mbar_arrive(&bar_sdp);  // S(n), dP(n) are in registers: step n + 1 may overwrite them
          if (!full) {  // hidden scores become -inf: exp2 of them is exactly 0, and so is dS
            // the visible columns as one bit mask per 32 columns, then one bit test and
            // select per score (cheaper than two compares per score)
#pragma unroll
            for (int q = 0; q < kEWCols / 32; ++q) {
              const int lo = min(max(vlo - 32 * q, 0), 32), hi = min(max(vhi - 32 * q + 1, 0), 32);
              const uint32_t below_hi = hi >= 32 ? 0xffffffffu : (1u << hi) - 1u;
              const uint32_t below_lo = lo >= 32 ? 0xffffffffu : (1u << lo) - 1u;
              const uint32_t m = below_hi & ~below_lo;
#pragma unroll
              for (int c = 0; c < 32; ++c) sv[32 * q + c] = ((m >> c) & 1u) ? sv[32 * q + c] : 0xFF800000u;
            }
          }
          const uint32_t row_off = static_cast<uint32_t>(hb * kBox + r * 128);
          // One 16-byte chunk (8 keys) of P and dS as bf16 pairs.
          auto chunk = [&](int q, uint32_t (&pw)[4], uint32_t (&dw)[4]) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c = 8 * q + 2 * e;
              float x0, x1, d0, d1;
              fma2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1]), a.scale_log2, -lse2, x0, x1);
              const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              sub_mul2(__uint_as_float(dpv[c]), __uint_as_float(dpv[c + 1]), dlt, p0, p1, d0, d1);
              pw[e] = pack_bf16x2(p0, p1);
              dw[e] = pack_bf16x2(d0, d1);
            }
          };
          auto store = [&](int q, const uint32_t (&pw)[4], const uint32_t (&dw)[4]) {
            const uint32_t sw = static_cast<uint32_t>((((qb + q) ^ (r & 7)) * 16));
            if (MODE == kDKV) st_shared_v4(p_s + row_off + sw, pw[0], pw[1], pw[2], pw[3]);
            st_shared_v4(ds_s + row_off + sw, dw[0], dw[1], dw[2], dw[3]);
          };
          if constexpr (!C::EARLY_S) {
            // S(n) was issued after step n - 1's accumulating products, so its
            // completion says the P / dS tiles are free: store as computed.
#pragma unroll
            for (int q = 0; q < NC; ++q) {
              uint32_t pw[4], dw[4];
              chunk(q, pw, dw);
              store(q, pw, dw);
            }
          } else {
            uint32_t pw[NC][4], dw[NC][4];
#pragma unroll
            for (int q = 0; q < NC; ++q) chunk(q, pw[q], dw[q]);
            // the previous step's accumulating products have read the P / dS tiles
            if (gs > 0) ok = __all_sync(0xffffffffu, mbar_wait(&bar_pfree, (gs - 1) & 1));
            if (!ok) break;
#pragma unroll
            for (int q = 0; q < NC; ++q) store(q, pw[q], dw[q]);
          }
        }
        fence_async_smem();  // the generic-proxy stores become visible to the tensor core
        tc_fence_before();
        mbar_arrive(&bar_p);
      }
      // ---- epilogue: the accumulators (rows = keys for dK, dV; query rows for dQ)
      if (ok && nsteps > 0) ok = __all_sync(0xffffffffu, mbar_wait(&bar_acc, nacc & 1));
      if (!ok) {
        if (lane == 0) set_status(a.status, MARS_DEV_TIMEOUT);
        break;
      } else {
        nacc += nsteps > 0;
        tc_fence_after();
        // The accumulator columns are split evenly over the warpgroups: dK then dV
        // (dKV mode) or dQ (dQ mode).  Warp (ew, quad) owns rows [32 quad, 32 quad + 32)
        // of the unit's tile and columns [c_lo, c_lo + SPAN) of accumulator m.
        constexpr int NACC = MODE == kDKV ? 2 : 1;
        constexpr int SPAN = NACC * D / kEW;  // columns per warpgroup, a multiple of 16
        static_assert(SPAN % 16 == 0 && D % SPAN == 0 && SPAN % 64 == 0 || MODE == kDQ, "accumulator split");
        const int m = (SPAN * ew) / D;
        const int c_lo = (SPAN * ew) % D;
        const float f = (MODE == kDKV && m == 1) ? 1.f : a.scale;  // dV carries no scale
        const bool fp32_out = MODE == kDKV && U.nch > 1;  // a chunk of a GQA group: its fp32 partial
        // The block leaves through shared memory, so that every global store writes
        // whole rows of consecutive addresses (a lane per row would scatter each store
        // instruction over 32 rows): the lane stages its row, 16-byte chunks XOR-swizzled
        // by the row, then the warp stores row after row.  The P / dS tiles are free
        // here (every product of the unit is complete): 8 KB per warp in dKV mode (P and
        // dS, 64 KB), 4 KB in dQ mode (dS, 32 KB).
        constexpr int STG = MODE == kDKV ? 8192 : 4096;
        static_assert(8 * STG <= (MODE == kDKV ? 4 : 2) * kBox && 2 * SPAN * 32 <= STG, "staging");
        const uint32_t stg = (MODE == kDKV ? p_s : ds_s) + static_cast<uint32_t>(warp - 2) * STG;
        // a staged block: 64 fp32 columns (256-byte rows) or all SPAN bf16 columns
        const int nblk = fp32_out ? SPAN / 64 : 1;
        const int cw = fp32_out ? 64 : SPAN;        // columns of a block
        const int rb = fp32_out ? 256 : 2 * SPAN;   // bytes of a staged row (<= 256)
        const int cpr = rb / 16;                    // 16-byte chunks per row: 4, 8 or 16
        const size_t plane = static_cast<size_t>(b) * (2 * a.L);
        for (int blk = 0; blk < nblk; ++blk) {
          const int c0 = c_lo + blk * cw;
          // W columns per batch of tensor-memory loads, awaited once
          constexpr int W = MODE == kDKV ? 64 : SPAN;
#pragma unroll 1
          for (int c = 0; c < cw; c += W) {
            uint32_t v[W];
#pragma unroll
            for (int x = 0; x < W; x += 32)
              tmem_ld32(tmem + lane_addr + C::ACC_COL + m * D + c0 + c + x, *reinterpret_cast<uint32_t(*)[32]>(&v[x]));
            tc_wait_ld();
            if (fp32_out) {
#pragma unroll
              for (int w = 0; w < W / 4; ++w) {
                const int ch = c / 4 + w;
                const uint32_t x0 = nsteps > 0 ? __float_as_uint(__uint_as_float(v[4 * w]) * f) : 0u;
                const uint32_t x1 = nsteps > 0 ? __float_as_uint(__uint_as_float(v[4 * w + 1]) * f) : 0u;
                const uint32_t x2 = nsteps > 0 ? __float_as_uint(__uint_as_float(v[4 * w + 2]) * f) : 0u;
                const uint32_t x3 = nsteps > 0 ? __float_as_uint(__uint_as_float(v[4 * w + 3]) * f) : 0u;
                st_shared_v4(stg + lane * rb + ((ch ^ (lane & (cpr - 1))) << 4), x0, x1, x2, x3);
              }
            } else {
#pragma unroll
              for (int w = 0; w < W / 8; ++w) {
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  pk[e] = nsteps > 0 ? pack_bf16x2(__uint_as_float(v[8 * w + 2 * e]) * f, __uint_as_float(v[8 * w + 2 * e + 1]) * f)
                                     : 0u;
                const int ch = c / 8 + w;
                st_shared_v4(stg + lane * rb + ((ch ^ (lane & (cpr - 1))) << 4), pk[0], pk[1], pk[2], pk[3]);
              }
            }
          }
          __syncwarp();
          // lane l stores chunk l % cpr of row j: 32 / cpr rows per instruction
          const int rpi = 32 / cpr;
#pragma unroll 1
          for (int j0 = 0; j0 < 32; j0 += rpi) {
            const int j = j0 + lane / cpr, ch = lane % cpr;
            const uint4 w4 = ld_shared_v4(stg + j * rb + ((ch ^ (j & (cpr - 1))) << 4));
            const int grow = u0 + quad * 32 + j;
            if (grow < uend) {
              if (fp32_out) {
                // the chunk's slot g G + chunk of the [2][b, 2L, Hq, D] partials
                float* dst = a.part + ((static_cast<size_t>(m) * a.batch * (2 * a.L) + plane + grow) * a.Hq +
                                       g * a.G + U.chunk) * D + c0;
                reinterpret_cast<uint4*>(dst)[ch] = w4;
              } else {
                uint16_t* base = MODE == kDKV ? (m == 0 ? a.dk : a.dv) : a.dq;
                const int H = MODE == kDKV ? a.Hkv : a.Hq;
                const int hout = MODE == kDKV ? g : hh;  // dKV: one chunk covers the whole group
                reinterpret_cast<uint4*>(base + ((plane + grow) * H + hout) * D + c0)[ch] = w4;
              }
            }
          }
          __syncwarp();
        }
        // Every elementwise warp has read its staged block before any of them writes
        // the next unit's P / dS into these tiles (a bounded wait, like every other).
        mbar_arrive(&bar_stg);
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_stg, nstg & 1));
        ++nstg;
        if (!ok) {
          if (lane == 0) set_status(a.status, MARS_DEV_TIMEOUT);
          break;
        }
      }
    }
  }
  if constexpr (MODE == kDQ) griddep_wait();
  griddep_launch_dependents();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// [batch, n, H, D] bf16 as a 4-D tensor loaded in [128 rows x 64 columns] SW128 boxes.
bool make_map(CUtensorMap* m, const void* ptr, int D, int H, int n, int batch) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(n),
                              static_cast<cuuint64_t>(batch)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2,
                                 static_cast<cuuint64_t>(n) * H * D * 2};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(kT), 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct OrderEntry {
  uint32_t code;  // tile | chunk << 16 | chunks << 24
  long long w;    // steps of one unit
};

// Cost, in steps, of the work a unit does besides its steps (the fixed tiles, the first
// products, the epilogue), and the extra for writing an fp32 partial instead of bf16.
constexpr long long kUnitCost = 2, kPartCost = 1;

// Steps until the last CTA of the dK/dV pass finishes when the persistent CTAs take
// the units in order, each as soon as it is free (each entry stands for per_entry units
// of equal weight).
long long makespan(const std::vector<OrderEntry>& es, long long per_entry, int sms) {
  std::priority_queue<long long, std::vector<long long>, std::greater<long long>> free_at;
  const long long units = static_cast<long long>(es.size()) * per_entry;
  for (long long i = 0; i < std::min<long long>(std::max(1, sms), units); ++i) free_at.push(0);
  long long end = 0;
  for (const OrderEntry& e : es) {
    const long long cost = e.w + kUnitCost + ((e.code >> 24) > 1 ? kPartCost : 0);
    for (long long u = 0; u < per_entry; ++u) {
      const long long t = free_at.top() + cost;
      free_at.pop();
      free_at.push(t);
      end = std::max(end, t);
    }
  }
  return end;
}

// Work units heaviest first.  Weight of a tile = the tiles on the other side it
// meets (per query head).  dKV: a tile's GQA group is split into chunks of query
// heads, because the heavy key tiles early in the clean stream are seen by most query
// tiles and a whole group in one unit would serialise on one SM; light tiles keep the
// whole group in one unit and need no partial.  A unit may hold at most a target
// number of steps, SM share / d for d in {1, 1.25, 1.5, 2, 2.5, 3, 4}; the chunking
// kept is the one whose heaviest-first schedule ends first (makespan), the fewest
// chunks on a tie.  The finishing time moves in steps as the chunk counts change,
// so no single d suits every shape.
bool make_order(const BwdArgs& a, int mode, int sms, UnitOrder* o, ChunkTable* ct) {
  const int n = 2 * a.nt;
  std::vector<long long> spt(n, 0);
  long long total = 0;
  for (int t = 0; t < n; ++t) {
    int lo[2] = {-1, -1}, hi[2] = {0, 0};
    for (int u = 0; u < n; ++u) {
      if (mode == kDKV ? tile_visible(a, u, t) : tile_visible(a, t, u)) {
        ++spt[t];
        const int st = u >= a.nt;
        if (lo[st] < 0) lo[st] = u;
        hi[st] = u + 1;
      }
    }
    if (lo[0] < 0) lo[0] = hi[0] = 0;  // empty clean range
    if (lo[1] < 0) lo[1] = hi[1] = n;  // empty noisy range
    // the visible tiles of each stream are one range (Eq. 2 is monotonic in the tile
    // index within a stream); the kernel relies on it
    if (spt[t] != (hi[0] - lo[0]) + (hi[1] - lo[1])) return false;
    o->rng[t][0] = static_cast<uint16_t>(lo[0]);
    o->rng[t][1] = static_cast<uint16_t>(hi[0]);
    o->rng[t][2] = static_cast<uint16_t>(lo[1]);
    o->rng[t][3] = static_cast<uint16_t>(hi[1]);
    total += spt[t];
  }
  auto build = [&](const std::vector<int>& nch, std::vector<OrderEntry>& es) {
    es.clear();
    for (int t = 0; t < n; ++t)
      for (int c = 0; c < nch[t]; ++c) {
        const int heads = mode == kDKV ? ((c + 1) * a.G) / nch[t] - (c * a.G) / nch[t] : 1;
        es.push_back({static_cast<uint32_t>(t) | (static_cast<uint32_t>(c) << 16) |
                          (static_cast<uint32_t>(nch[t]) << 24),
                      spt[t] * heads});
      }
    std::stable_sort(es.begin(), es.end(), [](const OrderEntry& x, const OrderEntry& y) { return x.w > y.w; });
  };
  std::vector<int> nch(n, 1);
  std::vector<OrderEntry> es;
  if (mode == kDKV) {
    const double share = static_cast<double>(total) * a.batch * a.Hq / std::max(1, sms);  // steps per SM
    const int gmax = std::min(a.G, 255);
    std::vector<int> cand(n);
    long long best = LLONG_MAX;
    for (const double d : {1.0, 1.25, 1.5, 2.0, 2.5, 3.0, 4.0}) {
      const long long target = std::max<long long>(1, static_cast<long long>(share / d));
      long long sum = 0;
      for (int t = 0; t < n; ++t) {
        const long long group = static_cast<long long>(a.G) * spt[t];
        cand[t] = static_cast<int>(std::min<long long>(gmax, std::max<long long>(1, (group + target - 1) / target)));
        sum += cand[t];
      }
      if (sum > kMaxEntries) std::fill(cand.begin(), cand.end(), 1);  // very long sequences: whole groups
      build(cand, es);
      const long long m = makespan(es, static_cast<long long>(a.batch) * a.Hkv, sms);
      if (m < best) {
        best = m;
        nch = cand;
      }
    }
    for (int t = 0; t < n; ++t) ct->nch[t] = static_cast<uint8_t>(nch[t]);
  }
  build(nch, es);
  o->n = static_cast<int>(es.size());
  for (int i = 0; i < o->n; ++i) o->entry[i] = es[i].code;
  return true;
}

template <int D, int MODE>
int launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
           const BwdArgs& a, const UnitOrder& order, cudaStream_t stream) {
  using C = BCfg<D, MODE>;
  auto big = bwd_kernel<D, MODE, kMaxEntries, kMaxTiles>;
  auto small = bwd_kernel<D, MODE, kSmallEntries, kSmallTiles>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(big, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(small, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return mars_host::cuda_fail(e);
    configured = true;
  }
  BwdArgs am = a;
  am.next_unit = a.next_unit + MODE;  // one counter per mode
  const long long units =
      static_cast<long long>(order.n) * (MODE == kDKV ? a.batch * a.Hkv : a.batch * a.Hq);
  const int grid = static_cast<int>(std::min<long long>(units, mars_host::num_sms()));  // persistent CTAs
  cudaLaunchConfig_t cfg = mars_host::pdl_config(dim3(grid), dim3(kThreads), C::SMEM, stream);
  cudaLaunchAttribute attr[1];
  mars_host::pdl_attr(cfg, attr);
  cudaError_t e;
  if (order.n <= kSmallEntries && 2 * a.nt <= kSmallTiles) {
    static SmallOrder so;  // filled and copied under the caller's lock
    std::copy(order.entry, order.entry + order.n, so.entry);
    for (int t = 0; t < 2 * a.nt; ++t) std::copy(order.rng[t], order.rng[t] + 4, so.rng[t]);
    so.n = order.n;
    e = cudaLaunchKernelEx(&cfg, small, tq, tk, tv, tdo, am, so);
  } else {
    e = cudaLaunchKernelEx(&cfg, big, tq, tk, tv, tdo, am, order);
  }
  return e == cudaSuccess ? MARS_OK : mars_host::cuda_fail(e);
}

inline size_t align_up(size_t x, size_t al) { return (x + al - 1) / al * al; }

}  // namespace

// Workspace: delta [b, Hq, 2L] fp32, the two work counters (256 bytes), then (GQA
// only) the dK | dV partials [2][b, 2L, Hq, D] fp32.
inline size_t delta_bytes(int batch, int L, int Hq) {
  return align_up(static_cast<size_t>(batch) * Hq * 2 * L * sizeof(float), 256);
}
constexpr size_t kCounterBytes = 256;

extern "C" size_t mars_train_attn_bwd_workspace_size(int batch, int L, int Hq, int Hkv, int D) {
  if (batch <= 0 || L <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0) return 0;
  const size_t part = Hq == Hkv ? 0 : 2 * static_cast<size_t>(batch) * 2 * L * Hq * D * sizeof(float);
  return delta_bytes(batch, L, Hq) + kCounterBytes + part;
}

extern "C" int mars_train_attn_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* o,
                                   const uint16_t* dout, const float* lse, uint16_t* dq, uint16_t* dk, uint16_t* dv,
                                   int batch, int L, int B, int Hq, int Hkv, int D, float scale, void* workspace,
                                   size_t workspace_bytes, int32_t* status, void* stream) {
  using mars_host::aligned16;
  MARS_HOST_CHECK(batch > 0 && L > 0 && B > 0 && Hq > 0 && Hkv > 0 && Hq % Hkv == 0, MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(D == 64 || D == 128, MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(scale > 0.f && scale < INFINITY, MARS_ERR_INVALID_ARG);
  const int nt = (L + kT - 1) / kT;
  MARS_HOST_CHECK(2 * nt <= kMaxTiles, MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(2LL * nt * batch * Hq < (1LL << 30), MARS_ERR_INVALID_ARG);
  const void* ptrs[] = {q, k, v, o, dout, dq, dk, dv};
  for (const void* p : ptrs) MARS_HOST_CHECK(p != nullptr && aligned16(p), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(lse != nullptr && mars_host::aligned4(lse), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(status == nullptr || mars_host::aligned4(status), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(workspace != nullptr && aligned16(workspace), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(workspace_bytes >= mars_train_attn_bwd_workspace_size(batch, L, Hq, Hkv, D),
                  MARS_ERR_WORKSPACE_TOO_SMALL);
  int rc = mars_host::check_device();
  if (rc != MARS_OK) return rc;

  BwdArgs a;
  a.lse = lse;
  a.delta = static_cast<const float*>(workspace);
  int* counters = reinterpret_cast<int*>(static_cast<char*>(workspace) + delta_bytes(batch, L, Hq));
  a.part = Hq == Hkv ? nullptr
                     : reinterpret_cast<float*>(static_cast<char*>(workspace) + delta_bytes(batch, L, Hq) +
                                                kCounterBytes);
  a.next_unit = counters;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.status = status;
  a.batch = batch;
  a.L = L;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = Hq / Hkv;
  a.nt = nt;
  a.scale_log2 = scale * kLog2e;
  a.scale = scale;
  CUtensorMap tq, tk, tv, tdo;
  if (!make_map(&tq, q, D, Hq, 2 * L, batch) || !make_map(&tk, k, D, Hkv, 2 * L, batch) ||
      !make_map(&tv, v, D, Hkv, 2 * L, batch) || !make_map(&tdo, dout, D, Hq, 2 * L, batch))
    return MARS_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int sms = mars_host::num_sms();
  // The orders depend only on the shape: the last shape's are kept.
  static UnitOrder order_kv, order_q;  // large: kept off the stack (calls on one thread at a time)
  static ChunkTable chunks;
  static int last_key[6] = {0, 0, 0, 0, 0, 0};
  static std::mutex order_mu;
  std::lock_guard<std::mutex> lock(order_mu);
  const int key[6] = {batch, L, B, Hq, Hkv, sms};
  if (!std::equal(key, key + 6, last_key)) {
    std::fill(last_key, last_key + 6, 0);
    if (!make_order(a, kDKV, sms, &order_kv, &chunks) || !make_order(a, kDQ, sms, &order_q, nullptr))
      return MARS_ERR_INVALID_ARG;
    std::copy(key, key + 6, last_key);
  }
  const long long rows = static_cast<long long>(batch) * 2 * L * Hq;
  {
    cudaLaunchConfig_t cfg = mars_host::pdl_config(dim3(static_cast<int>((rows * (D / 8) + 255) / 256)), dim3(256), 0, s);
    cudaLaunchAttribute attr[1];
    mars_host::pdl_attr(cfg, attr);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, delta_kernel, static_cast<const uint16_t*>(o),
                                             static_cast<const uint16_t*>(dout), static_cast<float*>(workspace),
                                             counters, batch, 2 * L, Hq, D);
    if (e != cudaSuccess) return mars_host::cuda_fail(e);
  }
  rc = D == 64 ? launch<64, kDKV>(tq, tk, tv, tdo, a, order_kv, s) : launch<128, kDKV>(tq, tk, tv, tdo, a, order_kv, s);
  if (rc != MARS_OK) return rc;
  if (a.part != nullptr) {
    const long long e8 = 2LL * batch * 2 * L * Hkv * D / 8;
    cudaLaunchConfig_t cfg = mars_host::pdl_config(dim3(static_cast<int>((e8 + 255) / 256)), dim3(256), 0, s);
    cudaLaunchAttribute attr[1];
    mars_host::pdl_attr(cfg, attr);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, reduce_kernel, static_cast<const float*>(a.part), dk, dv, batch, L,
                                             nt, Hkv, a.G, D, chunks);
    if (e != cudaSuccess) return mars_host::cuda_fail(e);
  }
  return D == 64 ? launch<64, kDQ>(tq, tk, tv, tdo, a, order_q, s) : launch<128, kDQ>(tq, tk, tv, tdo, a, order_q, s);
}
