// train_attn.cu - mars_train_attn: attention over z = [x ; x~] (length 2L)
// under the MARS structured mask.
//
// Method: "MARS: Enabling Autoregressive Models Multi-Token Generation",
// Sec. 3.2, Eq. 1 (concatenated clean / [MASK] streams) and Eq. 2 (mask):
// the clean half is causal; a placeholder of noisy block k sees the clean
// tokens of blocks < k and the placeholders of its own block up to itself.
//
// Structure that the kernel exploits: for every query row the visible keys
// form at most two intervals, one per stream,
//   clean row i:        clean [0, i]
//   noisy row t = i-L:  clean [0, B*floor(t/B) - 1]  and  noisy [L + B*floor(t/B), i]
// so a 128-row query tile (always inside one stream) only visits the key
// tiles that intersect those intervals: fully masked tiles are never loaded,
// tiles inside every row's interval take no mask, and the rest take the row's
// interval as one bit mask per 32 columns (one bit test per score).
//
// sm_103a design.  A work item is one 128-row query tile of one or two query
// heads that share a KV head (so both read the same K/V tiles); a host-side
// plan (longest first by a fitted cost model, then moves between CTAs) gives
// each persistent CTA (one per SM) its list of items.
//   warp 0      TMA producer: the item's Q tiles, then K and V tiles (SW128,
//               64-column boxes) into an NS-stage ring (full/empty mbarriers).
//   warp 1      TMEM owner and MMA issuer (one thread).  At D = 128 it issues
//               both query tiles' products; per key tile n the tensor pipe
//               runs, in issue order,
//                 PV_A(n), S_A(n+1) = Q_A K(n+1)^T, PV_B(n), S_B(n+1),
//               so while softmax warpgroup A works on S_A the tensor cores
//               compute B's products, and vice versa.  tcgen05 operations of
//               one thread execute in order, so S_X(n+1) overwrites the TMEM
//               columns that PV_X(n) reads only after PV_X(n) has read them,
//               and the commit after S_X(n+1) also covers PV_X(n).
//   warp 10     (D = 64 only) a second MMA issuer: warp 1 issues query tile
//               A's products and warp 10 tile B's, each in its own order
//               S_X(n+1), PV_X(n), so neither tile's chain waits on the
//               other's softmax (the issuing warps' own latency per wait and
//               issue was the step limit with one issuer).
//   warps 2..5  softmax warpgroup A, warps 6..9 warpgroup B (thread = query
//               row = TMEM lane): S from TMEM (on unmasked tiles with the
//               reducing load of sm_103a, which also returns the row max),
//               mask, row max, exp2; P is written to TMEM as bf16 pairs (over
//               S at D = 128, into its own columns at D = 64) and PV reads it
//               from there (the A operand of tcgen05.mma may live in TMEM).
//               On the partial tiles of the first query tile of each stream P
//               is also split into hi + lo bf16 terms (two PV passes): the rows
//               that see only a few keys, and so have no averaging to hide the
//               2^-9 rounding of a single bf16 P, all live there (every later
//               row sees at least ~B * floor(128 / B) keys).  O in TMEM is
//               rescaled only when the row max grows by more than 2^8 (lazy
//               rescaling); the epilogue normalises O and stores bf16 and the
//               log-sum-exp.
// Every mbarrier wait is bounded; a wait that gives up sets MARS_DEV_TIMEOUT
// in the status word and the role winds down without further waiting.
#include <cuda.h>

#include <algorithm>
#include <memory>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace {

using namespace mars;

constexpr int kBM = 128;        // query rows per query tile
constexpr int kBN = 128;        // keys per tile
constexpr int kBox = 128 * 128; // bytes of one [128 rows x 64 bf16] SW128 box
constexpr int kOBox = 32 * 128; // bytes of one [32 rows x 64 bf16] SW128 output box
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P values stay below 2^8
// Warps: TMA producer (warp 0), MMA issuer (warp 1), softmax warpgroups A
// (warps 2..5) and B (warps 6..9); at D = 64 a second MMA issuer (warp 10)
// serves warpgroup B.  Three warps share some SM sub-partitions, which caps the
// kernel at 168 registers per thread.
constexpr int kIssuerB = 10;

template <int D>
struct Cfg {
  static constexpr int NB = D / 64;  // 64-column boxes per row block
  static constexpr int NS = D == 64 ? 4 : 2;
  static constexpr int Q_BYTES = NB * kBox;   // one query tile
  static constexpr int KV_BYTES = NB * kBox;  // one K (or V) tile
  static constexpr int Q_OFF = 0;             // Q_A, Q_B
  static constexpr int K_OFF = Q_OFF + 2 * Q_BYTES;
  static constexpr int V_OFF = K_OFF + NS * KV_BYTES;
  static constexpr int O_OFF = V_OFF + NS * KV_BYTES;  // per softmax warp: one [32 rows x 64] SW128 box
  static constexpr int SMEM = O_OFF + 8 * kOBox + 1024;  // + slack to align the base to 1024
  static constexpr int TMEM_COLS = 512;
  // D = 64 keeps P apart from S (S_A | S_B | P_A | P_B | O_A | O_B), so the next S of a
  // warpgroup is computed while its softmax still works on the current tile.  At
  // D = 128 there is no room for it: P is written over S (S_A | S_B | O_A | O_B).
  static constexpr bool SEPP = D == 64;
  // SEPP: one MMA issuer per query tile (warps 1 and kIssuerB), each running its
  // own S and PV chain; the K/V stages and the Q tiles are released by both.
  static constexpr int THREADS = SEPP ? 32 * (kIssuerB + 1) : 320;
  static constexpr int RELEASES = SEPP ? 2 : 1;
  static constexpr int P_COL = 2 * kBN;  // P_x at P_COL + x * kBN / 2 (bf16 pairs), SEPP only
  static constexpr int O_COL = SEPP ? 3 * kBN : 2 * kBN;
  static_assert(!SEPP || O_COL + 2 * D <= TMEM_COLS, "tensor memory layout");
  static_assert(NS >= 2, "the next key tile is awaited before the current tile's stage is released");
};

struct TrainArgs {
  uint16_t* o;
  float* lse;
  int32_t* status;
  int batch, L, B, Hq, Hkv, G;
  float scale_log2;
  int nq;      // query tiles per stream
  int pairs;   // head slots per KV group: ceil(G / 2)
  int items;   // 2 * nq * batch * Hkv * pairs
  int planned; // 1: each CTA runs the item list the Plan gives it; 0: items blockIdx.x + n * gridDim.x
};

// Static schedule: CTA c runs items item[start[c] .. start[c+1]) in that order.  Built
// on the host by longest-processing-time-first list scheduling (item cost from its
// key-tile count), which keeps the persistent CTAs' loads within a few percent.
// The plan is a kernel parameter, copied with every launch: a launch of the kernel
// taking a 1,024-item plan (2.6 KB) starts ~1.2 us sooner than one taking the
// 8,192-item plan (17 KB), so the smaller is used whenever the items fit.
constexpr int kMaxPlanCtas = 256;
constexpr int kMaxPlanItems = 8192;
constexpr int kSmallPlanItems = 1024;
template <int CAP>
struct PlanT {
  uint16_t start[kMaxPlanCtas + 1];
  uint16_t item[CAP];
};
using Plan = PlanT<kMaxPlanItems>;
using SmallPlan = PlanT<kSmallPlanItems>;

// SW128 K-major / MN-major shared-memory matrix descriptor (tcgen05 format).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;  // descriptor version for sm_100-class tensor cores
  d |= 2ull << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor: bf16 x bf16 -> fp32, dense, M x N, A K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Key tiles visited by one query tile: n_clean clean tiles at 0, 128, ...
// (the first clean_full of them need no mask) then n_noisy noisy tiles
// starting at z position noisy_start.
struct Sched {
  int n_clean, clean_full, n_noisy, noisy_start;
  __host__ __device__ __forceinline__ int count() const { return n_clean + n_noisy; }
  __device__ __forceinline__ void at(int n, int& kstart, bool& noisy, bool& partial) const {
    if (n < n_clean) {
      kstart = kBN * n;
      noisy = false;
      partial = n >= clean_full;
    } else {
      kstart = noisy_start + kBN * (n - n_clean);
      noisy = true;
      partial = true;
    }
  }
};

__host__ __device__ __forceinline__ Sched make_sched(bool noisy_q, int j, int L, int B) {
  Sched s;
  if (!noisy_q) {
    const int rows_end = min(kBM * j + kBM, L);
    s.n_clean = (rows_end + kBN - 1) / kBN;
    s.clean_full = j;
    s.n_noisy = 0;
    s.noisy_start = 0;
  } else {
    const int t_min = kBM * j, t_max = min(kBM * j + kBM - 1, L - 1);
    const int c_lo = B * (t_min / B);   // clean prefix seen by every row of the tile
    const int c_hi = B * (t_max / B);   // clean prefix seen by the last row
    s.n_clean = (c_hi + kBN - 1) / kBN;
    s.clean_full = c_lo / kBN;
    s.noisy_start = L + c_lo;           // first placeholder any row of the tile sees
    s.n_noisy = (t_max - c_lo) / kBN + 1;
  }
  return s;
}

// One work item: query tile (noisy_q, j) of heads h_a and (when two_q) h_a + 1
// of batch b, sharing KV head g.  Items are numbered heaviest query tile first
// (noisy j, clean j for j = nq-1 .. 0), then batch / KV head / head pair.
struct Item {
  int b, g, h_a, j, r0, row_end;
  bool noisy_q, two_q;
  Sched sched;
};

__host__ __device__ __forceinline__ Item item_of(const TrainArgs& a, int idx) {
  Item it;
  const int per_rank = a.batch * a.Hkv * a.pairs;
  const int rank = idx / per_rank;
  int rest = idx % per_rank;
  const int pair = rest % a.pairs;
  rest /= a.pairs;
  it.g = rest % a.Hkv;
  it.b = rest / a.Hkv;
  it.h_a = it.g * a.G + 2 * pair;
  it.two_q = 2 * pair + 1 < a.G;
  it.j = a.nq - 1 - rank / 2;
  it.noisy_q = (rank & 1) == 0;
  it.r0 = it.noisy_q ? a.L + kBM * it.j : kBM * it.j;
  it.row_end = it.noisy_q ? 2 * a.L : a.L;
  it.sched = make_sched(it.noisy_q, it.j, a.L, a.B);
  return it;
}

// The n-th item of this CTA, or -1 past its last.
template <int CAP>
__device__ __forceinline__ int nth_item(const PlanT<CAP>& p, const TrainArgs& a, int n) {
  if (a.planned) {
    const int j = p.start[blockIdx.x] + n;
    return j < p.start[blockIdx.x + 1] ? p.item[j] : -1;
  }
  const int idx = blockIdx.x + n * gridDim.x;
  return idx < a.items ? idx : -1;
}

template <int D, int CAP>
__global__ void __launch_bounds__(Cfg<D>::THREADS, 1)
    train_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                      const TrainArgs a, const __grid_constant__ PlanT<CAP> plan) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar_q_full, bar_q_empty, bar_k[C::NS], bar_v[C::NS], bar_kv_empty[C::NS],
      bar_s[2], bar_p[2], bar_o[2], bar_sfree[2], bar_pfree[2];
  __shared__ uint32_t tmem_slot;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bar_q_full, 1);
    mbar_init(&bar_q_empty, C::RELEASES);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&bar_k[s], 1);
      mbar_init(&bar_v[s], 1);
      mbar_init(&bar_kv_empty[s], C::RELEASES);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bar_s[x], 1);
      mbar_init(&bar_p[x], 128);
      mbar_init(&bar_o[x], 1);
      mbar_init(&bar_sfree[x], 128);  // SEPP: S_x has been read into registers
      mbar_init(&bar_pfree[x], 1);    // SEPP: the PV that read P_x is complete
    }
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  // launched as a programmatic dependent: set-up above overlaps the previous kernel,
  // nothing global is touched before it has completed
  griddep_wait();

  const uint32_t q_s = smem_u32(smem + C::Q_OFF);
  const uint32_t k_s = smem_u32(smem + C::K_OFF);
  const uint32_t v_s = smem_u32(smem + C::V_OFF);

  if (warp == 0) {
    // ================= TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int kt = 0, t = 0;  // CTA-local key-tile and item counters
      for (int idx; (idx = nth_item(plan, a, t)) >= 0; ++t) {
        const Item it = item_of(a, idx);
        if (t > 0 && !mbar_wait(&bar_q_empty, (t - 1) & 1)) {
          set_status(a.status, MARS_DEV_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(&bar_q_full, (it.two_q ? 2 : 1) * C::Q_BYTES);
        for (int c = 0; c < C::NB; ++c) {
          tma_load_4d(q_s + c * kBox, &tm_q, &bar_q_full, 64 * c, it.h_a, it.r0, it.b);
          if (it.two_q) tma_load_4d(q_s + C::Q_BYTES + c * kBox, &tm_q, &bar_q_full, 64 * c, it.h_a + 1, it.r0, it.b);
        }
        bool ok = true;
        for (int n = 0; n < it.sched.count(); ++n, ++kt) {
          const int st = kt % C::NS;
          if (kt >= C::NS && !mbar_wait(&bar_kv_empty[st], ((kt / C::NS) - 1) & 1)) {
            set_status(a.status, MARS_DEV_TIMEOUT);
            ok = false;
            break;
          }
          int kstart;
          bool nz, part;
          it.sched.at(n, kstart, nz, part);
          // SEPP: K and V of the stage both complete bar_k (one wait before its S);
          // otherwise V has its own barrier, awaited just before the PV
          uint64_t* bv = C::SEPP ? &bar_k[st] : &bar_v[st];
          mbar_arrive_expect_tx(&bar_k[st], C::SEPP ? 2 * C::KV_BYTES : C::KV_BYTES);
          for (int c = 0; c < C::NB; ++c)
            tma_load_4d(k_s + st * C::KV_BYTES + c * kBox, &tm_k, &bar_k[st], 64 * c, it.g, kstart, it.b);
          if (!C::SEPP) mbar_arrive_expect_tx(bv, C::KV_BYTES);
          for (int c = 0; c < C::NB; ++c)
            tma_load_4d(v_s + st * C::KV_BYTES + c * kBox, &tm_v, bv, 64 * c, it.g, kstart, it.b);
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (C::SEPP && (warp == 1 || warp == kIssuerB)) {
    // ================= MMA issuer of query tile X (SEPP).  The whole warp runs the
    // schedule, so the descriptors stay warp-uniform; one elected lane issues the
    // tcgen05 operations and their commits (a commit tracks its own thread's MMAs,
    // and one thread's tcgen05 operations execute in issue order).  Per key tile n:
    //   S_X(n + 1) = Q_X K(n + 1)^T once softmax X has read S_X(n), then
    //   PV_X(n) once softmax X has stored P_X(n);
    // the stage of K/V(n) and the Q tiles are released by a commit of each issuer
    // (barriers of count 2).  Issuer B takes no part in an item with one query tile
    // beyond releasing what it would have released.
    const bool leader = elect_one();
    const int X = warp == 1 ? 0 : 1;
    constexpr uint32_t id_qk = idesc_bf16(kBM, kBN, false);
    constexpr uint32_t id_pv = idesc_bf16(kBM, D, true);
    const uint64_t desc_q = smem_desc(q_s + X * C::Q_BYTES, 16, 1024), desc_k = smem_desc(k_s, 16, 1024);
    const uint64_t desc_v = smem_desc(v_s, kBox, 1024);
    const uint32_t s_tm = tmem + X * kBN;
    const uint32_t p_tm = tmem + C::P_COL + X * (kBN / 2);
    const uint32_t o_tm = tmem + C::O_COL + X * D;
    int kt = 0, gs = 0, cp = 0;  // key tiles, S products issued, P phases consumed
    bool ok = true;
    auto wait_all = [&](uint64_t* bar, int parity) { ok = ok && __all_sync(0xffffffffu, mbar_wait(bar, parity)); };
    auto issue_s = [&](int st) {
      if (gs > 0) {
        wait_all(&bar_sfree[X], (gs - 1) & 1);
        if (!ok) return;
        tc_fence_after();
      }
      ++gs;
      const uint64_t kb = desc_k + ((st * C::KV_BYTES) >> 4);
      if (leader) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = ((ks >> 2) * kBox + (ks & 3) * 32) >> 4;
          tc_mma_ss(s_tm, desc_q + off, kb + off, id_qk, ks > 0 ? 1u : 0u);
        }
        tc_commit(&bar_s[X]);
      }
      __syncwarp();
    };
    auto issue_pv = [&](int st, bool first, bool split) {
      const uint64_t vb = desc_v + ((st * C::KV_BYTES) >> 4);
      for (int part = 0; part < (split ? 2 : 1); ++part) {
        wait_all(&bar_p[X], cp & 1);
        if (!ok) return;
        ++cp;
        tc_fence_after();
        if (leader) {
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks)
            tc_mma_ts(o_tm, p_tm + ks * 8, vb + ((ks * 16 * 128) >> 4), id_pv,
                      (first && part == 0 && ks == 0) ? 0u : 1u);
          tc_commit(&bar_pfree[X]);
        }
        __syncwarp();
      }
    };
    for (int t = 0, idx; ok && (idx = nth_item(plan, a, t)) >= 0; ++t) {
      const Item it = item_of(a, idx);
      const int nt = it.sched.count();
      wait_all(&bar_q_full, t & 1);
      if (!ok) break;
      if (X == 1 && !it.two_q) {
        // nothing to compute: release the Q tiles and each K/V stage once it is
        // filled (a release before the fill would count toward the previous phase)
        if (leader) mbar_arrive(&bar_q_empty);
        for (int n = 0; ok && n < nt; ++n, ++kt) {
          wait_all(&bar_k[kt % C::NS], (kt / C::NS) & 1);
          if (ok && leader) mbar_arrive(&bar_kv_empty[kt % C::NS]);
        }
        __syncwarp();
        continue;
      }
      wait_all(&bar_k[kt % C::NS], (kt / C::NS) & 1);
      if (!ok) break;
      tc_fence_after();
      issue_s(kt % C::NS);
      if (!ok) break;
      if (nt == 1 && leader) tc_commit(&bar_q_empty);
      for (int n = 0; ok && n < nt; ++n, ++kt) {
        const int st = kt % C::NS, st1 = (kt + 1) % C::NS;
        const bool last = n + 1 == nt;
        int kstart;
        bool nz, part;
        it.sched.at(n, kstart, nz, part);
        const bool split = part && it.j == 0;  // same rule as the softmax warps
        if (!last) {
          wait_all(&bar_k[st1], ((kt + 1) / C::NS) & 1);
          if (!ok) break;
          tc_fence_after();
          issue_s(st1);
          if (!ok) break;
          if (n + 2 == nt && leader) tc_commit(&bar_q_empty);  // the item's last S product is issued
        }
        issue_pv(st, n == 0, split);  // V(n) arrived with K(n), awaited before S(n)
        if (!ok) break;
        if (leader) {
          if (last) tc_commit(&bar_o[X]);
          tc_commit(&bar_kv_empty[st]);
        }
        __syncwarp();
      }
    }
    if (!ok && leader) set_status(a.status, MARS_DEV_TIMEOUT);
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer (D = 128).  The whole warp runs the schedule, so the
    // descriptors stay warp-uniform; one elected lane issues the tcgen05
    // operations and their commits (a commit tracks its own thread's MMAs).
    {
      const bool leader = elect_one();
      constexpr uint32_t id_qk = idesc_bf16(kBM, kBN, false);
      constexpr uint32_t id_pv = idesc_bf16(kBM, D, true);
      int kt = 0, t = 0;
      int cp[2] = {0, 0};  // P-ready phases consumed per query tile
      bool ok = true;
      // Descriptor start addresses are in 16-byte units (bits 0..13), so stepping
      // a descriptor by `bytes` adds bytes >> 4 to its low word.
      const uint64_t desc_q = smem_desc(q_s, 16, 1024), desc_k = smem_desc(k_s, 16, 1024);
      const uint64_t desc_v = smem_desc(v_s, kBox, 1024);
      auto wait_all = [&](uint64_t* bar, int parity) {
        ok = ok && __all_sync(0xffffffffu, mbar_wait(bar, parity));
      };
      auto commit = [&](uint64_t* bar) {
        if (leader) tc_commit(bar);
      };
      auto issue_qk = [&](int x, int st) {
        const uint64_t qa = desc_q + ((x * C::Q_BYTES) >> 4);
        const uint64_t kb = desc_k + ((st * C::KV_BYTES) >> 4);
        if (leader) {
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = ((ks >> 2) * kBox + (ks & 3) * 32) >> 4;
            tc_mma_ss(tmem + x * kBN, qa + off, kb + off, id_qk, ks > 0 ? 1u : 0u);
          }
          tc_commit(&bar_s[x]);
        }
        __syncwarp();
      };
      auto issue_pv = [&](int x, int st, bool first, bool split) {
        wait_all(&bar_p[x], cp[x] & 1);
        if (!ok) return;
        ++cp[x];
        tc_fence_after();
        const uint32_t s_col = tmem + x * kBN;  // P over the columns of S_x
        const uint32_t o_col = tmem + C::O_COL + x * D;
        const uint64_t vb = desc_v + ((st * C::KV_BYTES) >> 4);
        if (leader) {
          if (!split) {
#pragma unroll
            for (int ks = 0; ks < kBN / 16; ++ks)
              tc_mma_ts(o_col, s_col + ks * 8, vb + ((ks * 16 * 128) >> 4), id_pv, (!first || ks > 0) ? 1u : 0u);
          } else {
            // keys [16 ks, 16 ks + 16): hi at column 32 (ks / 2) + 8 (ks % 2), lo 16 columns later
#pragma unroll
            for (int ks = 0; ks < kBN / 16; ++ks) {
              const uint32_t pc = s_col + 32 * (ks >> 1) + 8 * (ks & 1);
              tc_mma_ts(o_col, pc, vb + ((ks * 16 * 128) >> 4), id_pv, (!first || ks > 0) ? 1u : 0u);
              tc_mma_ts(o_col, pc + 16, vb + ((ks * 16 * 128) >> 4), id_pv, 1u);
            }
          }
        }
        __syncwarp();
      };
      for (int idx; ok && (idx = nth_item(plan, a, t)) >= 0; ++t) {
        const Item it = item_of(a, idx);
        const int nt = it.sched.count();
        wait_all(&bar_q_full, t & 1);
        // prologue: S(0) for both query tiles
        wait_all(&bar_k[kt % C::NS], (kt / C::NS) & 1);
        if (!ok) break;
        tc_fence_after();
        issue_qk(0, kt % C::NS);
        if (it.two_q) issue_qk(1, kt % C::NS);
        if (nt == 1) commit(&bar_q_empty);
        for (int n = 0; ok && n < nt; ++n, ++kt) {
          const int st = kt % C::NS, st1 = (kt + 1) % C::NS;
          const bool last = n + 1 == nt;
          int kstart;
          bool nz, part;
          it.sched.at(n, kstart, nz, part);
          const bool split = part && it.j == 0;  // same rule as the softmax warps
          wait_all(&bar_v[st], (kt / C::NS) & 1);
          if (!ok) break;
          issue_pv(0, st, n == 0, split);
          if (!ok) break;
          if (last) commit(&bar_o[0]);
          if (!last) {
            wait_all(&bar_k[st1], ((kt + 1) / C::NS) & 1);
            if (!ok) break;
            tc_fence_after();
            issue_qk(0, st1);
          }
          if (it.two_q) {
            issue_pv(1, st, n == 0, split);
            if (!ok) break;
            if (last) commit(&bar_o[1]);
            if (!last) issue_qk(1, st1);
          }
          if (n + 2 == nt) commit(&bar_q_empty);  // the item's last S products are issued
          commit(&bar_kv_empty[st]);
        }
      }
      if (!ok && leader) set_status(a.status, MARS_DEV_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ================= softmax / epilogue: warpgroup x = 0 (warps 2..5) or 1 (warps 6..9)
    const int x = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_col = tmem + lane_addr + x * kBN;
    const uint32_t o_col = tmem + lane_addr + C::O_COL + x * D;
    int cs = 0, co = 0;  // S-ready and O-ready phases consumed
    int cpw = 0;         // P_x writes (SEPP), one per P-ready phase
    bool ok = true;
    for (int t = 0, idx; ok && (idx = nth_item(plan, a, t)) >= 0; ++t) {
      const Item it = item_of(a, idx);
      if (x == 1 && !it.two_q) continue;
      const int h = it.h_a + x;
      const int i = it.r0 + r;  // z position of this row
      // visible key intervals of this row: clean [0, c_hi_v], noisy [n_lo_v, n_hi_v]
      int c_hi_v, n_lo_v, n_hi_v;
      if (i < a.L) {
        c_hi_v = i;
        n_lo_v = 1;
        n_hi_v = 0;
      } else {
        const int tt = i - a.L;
        const int c = a.B * (tt / a.B);
        c_hi_v = c - 1;
        n_lo_v = a.L + c;
        n_hi_v = i;
      }
      float m_used = -INFINITY;  // max the current P values are relative to
      float l = 0.f;
      const int nt = it.sched.count();
      for (int n = 0; n < nt; ++n) {
        int kstart;
        bool nz, part;
        it.sched.at(n, kstart, nz, part);
        const bool split = part && it.j == 0;  // rows that see few keys in total live only here
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_s[x], cs & 1));
        if (!ok) break;
        ++cs;
        tc_fence_after();
        // visible columns of this row inside the tile: [vlo, vhi] (empty when vlo > vhi)
        const int vlo = part ? max((nz ? n_lo_v : 0) - kstart, 0) : 0;
        const int vhi = part ? min((nz ? n_hi_v : c_hi_v) - kstart, kBN - 1) : kBN - 1;
        if constexpr (C::SEPP) {
          // The noisy tile of the query tile's own blocks (its last tile, at L + 128 j):
          // row r sees only the keys [B floor(r / B), r] of the tile, at most B of them,
          // and when B divides 32 they all lie in the row's warp's own 32 columns.  Only
          // those 32 scores are read, masked and exponentiated; the other 96 columns of
          // P are stored as zeros.  (Not on split tiles: j = 0 keeps the hi + lo P.)
          const bool self_tile = it.noisy_q && it.j > 0 && n == nt - 1 && (32 % a.B) == 0 &&
                                 kstart == a.L + kBM * it.j;
          if (self_tile) {
            uint32_t v[32];
            tmem_ld32(s_col + 32 * quad, v);
            tc_wait_ld();
            tc_fence_before();
            mbar_arrive(&bar_sfree[x]);  // S_x is in registers: the next S may overwrite it
            {
              const int lo = min(max(vlo - 32 * quad, 0), 32), hi = min(max(vhi - 32 * quad + 1, 0), 32);
              const uint32_t below_hi = hi >= 32 ? 0xffffffffu : (1u << hi) - 1u;
              const uint32_t below_lo = lo >= 32 ? 0xffffffffu : (1u << lo) - 1u;
              const uint32_t msk = below_hi & ~below_lo;
#pragma unroll
              for (int c = 0; c < 32; ++c) v[c] = ((msk >> c) & 1u) ? v[c] : 0xFF800000u;
            }
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
              mx0 = fmax3(mx0, __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
              mx1 = fmax3(mx1, __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
            }
            const float tmax = fmaxf(mx0, mx1) * a.scale_log2;
            float alpha = 1.f;
            const bool grow = tmax > m_used + kRescaleThreshold;
            if (grow) {
              alpha = fast_exp2(m_used - tmax);  // 0 when m_used is -inf
              m_used = tmax;
            }
            const float neg_mu = m_used == -INFINITY ? 0.f : -m_used;
            uint64_t sum2x = 0;
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float x0, x1;
              fma2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]), a.scale_log2, neg_mu, x0, x1);
              const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              add2(sum2x, p0, p1);
              pk[e] = pack_bf16x2(p0, p1);
            }
            if (cpw > 0) {
              ok = __all_sync(0xffffffffu, mbar_wait(&bar_pfree[x], (cpw - 1) & 1));
              if (!ok) break;
            }
            tc_fence_after();
            if (n > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll 1
              for (int c = 0; c < D; c += 16) {
                uint32_t ov[16];
                tmem_ld16(o_col + c, ov);
                tc_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                tmem_st16(o_col + c, ov);
              }
            }
            const uint32_t p_col = tmem + lane_addr + C::P_COL + x * (kBN / 2);
            uint32_t zero[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) zero[e] = 0u;
#pragma unroll
            for (int q = 0; q < kBN / 32; ++q) {  // keys [32 q, 32 q + 32) -> columns [16 q, 16 q + 16)
              if (q == quad)
                tmem_st16(p_col + 16 * q, pk);
              else
                tmem_st16(p_col + 16 * q, zero);
            }
            l = l * alpha + sum2(sum2x);
            tc_wait_st();
            tc_fence_before();
            mbar_arrive(&bar_p[x]);
            ++cpw;
            continue;
          }
        }
        // One pass: the row's 128 scores are read from tensor memory once and kept in
        // registers for the max and then exp2 and the bf16 store of P.  An unmasked tile
        // reads them with the reducing load, which also returns each 32 columns' maximum;
        // a masked tile turns hidden scores into -inf (exp2 of them is exactly 0) and
        // takes the maximum after that.
        uint32_t v0[kBN];
        float gmax[kBN / 32];
        if (!part) {
#pragma unroll
          for (int c = 0; c < kBN; c += 32)
            gmax[c / 32] = tmem_ld32_max(s_col + c, *reinterpret_cast<uint32_t(*)[32]>(&v0[c]));
        } else {
#pragma unroll
          for (int c = 0; c < kBN; c += 32) tmem_ld32(s_col + c, *reinterpret_cast<uint32_t(*)[32]>(&v0[c]));
        }
        tc_wait_ld();
        if constexpr (C::SEPP) {
          tc_fence_before();
          mbar_arrive(&bar_sfree[x]);  // S_x is in registers: the next S may overwrite it
        }
        float tile_max;
        if (!part) {
          static_assert(kBN == 128, "four reducing loads per tile");
          tile_max = fmaxf(fmaxf(gmax[0], gmax[1]), fmaxf(gmax[2], gmax[3])) * a.scale_log2;
        } else {
          // the row's visible columns as one bit mask per 32 columns, then one bit
          // test and select per score (cheaper than two compares per score)
#pragma unroll
          for (int q = 0; q < kBN / 32; ++q) {
            const int lo = min(max(vlo - 32 * q, 0), 32), hi = min(max(vhi - 32 * q + 1, 0), 32);
            const uint32_t below_hi = hi >= 32 ? 0xffffffffu : (1u << hi) - 1u;
            const uint32_t below_lo = lo >= 32 ? 0xffffffffu : (1u << lo) - 1u;
            const uint32_t m = below_hi & ~below_lo;
#pragma unroll
            for (int c = 0; c < 32; ++c) v0[32 * q + c] = ((m >> c) & 1u) ? v0[32 * q + c] : 0xFF800000u;
          }
          float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
          for (int c = 0; c < kBN; c += 8) {
            mx0 = fmax3(mx0, __uint_as_float(v0[c]), __uint_as_float(v0[c + 1]));
            mx1 = fmax3(mx1, __uint_as_float(v0[c + 2]), __uint_as_float(v0[c + 3]));
            mx2 = fmax3(mx2, __uint_as_float(v0[c + 4]), __uint_as_float(v0[c + 5]));
            mx3 = fmax3(mx3, __uint_as_float(v0[c + 6]), __uint_as_float(v0[c + 7]));
          }
          tile_max = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * a.scale_log2;
        }
        // lazy rescale: keep the old reference max unless the new one is 2^8 larger.
        // PV_x(n-1) is complete here: S_x(n) was issued after it and its commit covers it.
        float alpha = 1.f;
        const bool grow = tile_max > m_used + kRescaleThreshold;
        if (grow) {
          alpha = fast_exp2(m_used - tile_max);  // 0 when m_used is -inf
          m_used = tile_max;
        }
        auto rescale_o = [&]() {
#pragma unroll 1
          for (int c = 0; c < D; c += 16) {
            uint32_t ov[16];
            tmem_ld16(o_col + c, ov);
            tc_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st16(o_col + c, ov);
          }
        };
        const float neg_mu = m_used == -INFINITY ? 0.f : -m_used;
        if constexpr (C::SEPP) {
          // P in registers first (PV_x of the previous tile may still be reading P_x),
          // then wait for that PV, rescale O if the max grew, and store P_x: keys
          // [32q, 32q + 32) -> columns [16q, 16q + 16).  A split tile stores hi, waits for
          // its PV, then stores lo.
          const uint32_t p_col = tmem + lane_addr + C::P_COL + x * (kBN / 2);
          uint64_t sum2x = 0;
          if (!split) {
            uint32_t hi[kBN / 2];
#pragma unroll
            for (int e = 0; e < kBN / 2; ++e) {
              float x0, x1;
              fma2(__uint_as_float(v0[2 * e]), __uint_as_float(v0[2 * e + 1]), a.scale_log2, neg_mu, x0, x1);
              const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              add2(sum2x, p0, p1);
              hi[e] = pack_bf16x2(p0, p1);
            }
            if (cpw > 0) {
              ok = __all_sync(0xffffffffu, mbar_wait(&bar_pfree[x], (cpw - 1) & 1));
              if (!ok) break;
            }
            tc_fence_after();
            if (n > 0 && __any_sync(0xffffffffu, grow)) rescale_o();
#pragma unroll
            for (int q = 0; q < kBN / 32; ++q)
              tmem_st16(p_col + 16 * q, *reinterpret_cast<uint32_t(*)[16]>(&hi[16 * q]));
          } else {
            if (cpw > 0) {
              ok = __all_sync(0xffffffffu, mbar_wait(&bar_pfree[x], (cpw - 1) & 1));
              if (!ok) break;
            }
            tc_fence_after();
            if (n > 0 && __any_sync(0xffffffffu, grow)) rescale_o();
            uint32_t lo[kBN / 2];
#pragma unroll
            for (int q = 0; q < kBN / 32; ++q) {
              uint32_t hq[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                float x0, x1;
                fma2(__uint_as_float(v0[32 * q + 2 * e]), __uint_as_float(v0[32 * q + 2 * e + 1]), a.scale_log2,
                     neg_mu, x0, x1);
                const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                add2(sum2x, p0, p1);
                hq[e] = pack_bf16x2(p0, p1);
                lo[16 * q + e] = pack_bf16x2(p0 - bf16lo_to_f32(hq[e]), p1 - bf16hi_to_f32(hq[e]));
              }
              tmem_st16(p_col + 16 * q, hq);
            }
            tc_wait_st();
            tc_fence_before();
            mbar_arrive(&bar_p[x]);  // hi
            ++cpw;
            ok = __all_sync(0xffffffffu, mbar_wait(&bar_pfree[x], (cpw - 1) & 1));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int q = 0; q < kBN / 32; ++q)
              tmem_st16(p_col + 16 * q, *reinterpret_cast<uint32_t(*)[16]>(&lo[16 * q]));
          }
          l = l * alpha + sum2(sum2x);
          tc_wait_st();
          tc_fence_before();
          mbar_arrive(&bar_p[x]);  // P (non-split) or lo (split)
          ++cpw;
          continue;
        }
        if (n > 0 && __any_sync(0xffffffffu, grow)) rescale_o();
        // P = exp2(s * scale_log2 - mu) as bf16 pairs, written over S columns already read:
        // keys [32q, 32q + 32) -> hi in columns [16q, 16q + 16); on split tiles hi in
        // [32q, 32q + 16) and lo = P - hi in [32q + 16, 32q + 32).
        uint64_t sum2x = 0;  // two fp32 partial sums (bits of +0.0f)
#pragma unroll
        for (int q = 0; q < kBN / 32; ++q) {
          if (!split) {
            uint32_t hi[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float x0, x1;
              fma2(__uint_as_float(v0[32 * q + 2 * e]), __uint_as_float(v0[32 * q + 2 * e + 1]), a.scale_log2,
                   neg_mu, x0, x1);
              const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              add2(sum2x, p0, p1);
              hi[e] = pack_bf16x2(p0, p1);
            }
            tmem_st16(s_col + 16 * q, hi);
          } else {
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float x0, x1;
              fma2(__uint_as_float(v0[32 * q + 2 * e]), __uint_as_float(v0[32 * q + 2 * e + 1]), a.scale_log2,
                   neg_mu, x0, x1);
              const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              add2(sum2x, p0, p1);
              hi[e] = pack_bf16x2(p0, p1);
              lo[e] = pack_bf16x2(p0 - bf16lo_to_f32(hi[e]), p1 - bf16hi_to_f32(hi[e]));
            }
            tmem_st16(s_col + 32 * q, hi);
            tmem_st16(s_col + 32 * q + 16, lo);
          }
        }
        l = l * alpha + sum2(sum2x);
        tc_wait_st();
        tc_fence_before();
        mbar_arrive(&bar_p[x]);
      }
      if (!ok) break;

      // ---- epilogue: O / l -> bf16, log-sum-exp
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_o[x], co & 1));
      if (!ok) break;
      ++co;
      tc_fence_after();
      const float inv = 1.f / l;
      const bool store = i < it.row_end;
      // O / l as bf16 -> this warp's [32 rows x 64] SW128 box in shared memory -> TMA
      // store, one 64-column box at a time.  The store map views O as
      // [2 * batch, L, Hq, D] so rows past the end of the stream are not written.
      const uint32_t obox = smem_u32(smem + C::O_OFF) + (x * 4 + quad) * kOBox;
      const uint32_t orow = obox + lane * 128;
#pragma unroll 1
      for (int bx = 0; bx < C::NB; ++bx) {
        uint32_t ov[64];
        tmem_ld32(o_col + 64 * bx, *reinterpret_cast<uint32_t(*)[32]>(&ov[0]));
        tmem_ld32(o_col + 64 * bx + 32, *reinterpret_cast<uint32_t(*)[32]>(&ov[32]));
        if (lane == 0) bulk_wait_read_all();  // the previous store out of this box has read it
        __syncwarp();
        tc_wait_ld();
#pragma unroll
        for (int c16 = 0; c16 < 8; ++c16) {
          const uint32_t* f = &ov[8 * c16];
          const uint32_t w0 = pack_bf16x2(__uint_as_float(f[0]) * inv, __uint_as_float(f[1]) * inv);
          const uint32_t w1 = pack_bf16x2(__uint_as_float(f[2]) * inv, __uint_as_float(f[3]) * inv);
          const uint32_t w2 = pack_bf16x2(__uint_as_float(f[4]) * inv, __uint_as_float(f[5]) * inv);
          const uint32_t w3 = pack_bf16x2(__uint_as_float(f[6]) * inv, __uint_as_float(f[7]) * inv);
          st_shared_v4(orow + ((c16 ^ (lane & 7)) << 4), w0, w1, w2, w3);
        }
        fence_async_smem();
        __syncwarp();
        const int row0 = it.r0 - (it.noisy_q ? a.L : 0) + 32 * quad;  // first row of the box in its stream
        if (lane == 0 && row0 < a.L) {
          tma_store_4d(&tm_o, obox, 64 * bx, h, row0, 2 * it.b + (it.noisy_q ? 1 : 0));
          bulk_commit_group();
        }
      }
      if (store && a.lse != nullptr)
        a.lse[(static_cast<size_t>(it.b) * a.Hq + h) * 2 * a.L + i] = (m_used + __log2f(l)) * 0.6931471805599453f;
      tc_fence_before();
    }
    if (lane == 0) bulk_wait_all();  // output stores complete before the CTA exits
    if (!ok && lane == 0) set_status(a.status, MARS_DEV_TIMEOUT);
  }

  griddep_launch_dependents();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
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

// [batch, n, H, D] bf16 viewed as a 4-D tensor with 64-column x box_rows SW128 boxes.
bool make_map(CUtensorMap* m, const void* ptr, int D, int H, int n, int batch, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(n),
                              static_cast<cuuint64_t>(batch)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2,
                                 static_cast<cuuint64_t>(n) * H * D * 2};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Work plan for (shape, grid), cached.  Item cost model, fitted by least squares to
// per-item durations measured on GB300 (globaltimer at each item's epilogue, both
// training shapes; 7-8% rms error per item), in units of 0.01 us:
//   key tiles x (two query tiles ? c2 : c1) + partial tiles of a one-head item x p1
//   + per item o + (first query tile of a stream: the hi/lo split) key tiles x sp.
// Items are assigned longest-processing-time first, then the most loaded CTA gives
// up an item (or trades one for a cheaper one) while that lowers its load: with only
// ~3-4 items per CTA, LPT alone leaves the slowest CTA ~10% above the mean.
struct CostModel {
  int c2, c1, p1, o, sp;
};
constexpr CostModel kCost64 = {160, 91, 52, 27, 94};
constexpr CostModel kCost128 = {176, 139, 86, 15, 132};

struct PlanEntry {
  long long key[8];
  std::unique_ptr<Plan> plan;
  std::unique_ptr<SmallPlan> small;  // the same plan when the items fit
};
std::mutex& plan_mutex() {
  static std::mutex mu;
  return mu;
}

// The cached plan of (shape, grid), or nullptr (no plan: items round-robin).  The
// caller holds plan_mutex() until its launch has copied the plan.
const PlanEntry* plan_for(const TrainArgs& a, int D, int grid) {
  if (grid > kMaxPlanCtas || a.items > kMaxPlanItems) return nullptr;
  static std::vector<PlanEntry> cache;
  const long long key[8] = {a.batch, a.L, a.B, a.Hq, a.Hkv, D, grid, 0};
  for (const PlanEntry& e : cache)
    if (std::equal(key, key + 8, e.key)) return &e;
  const CostModel cm = D == 64 ? kCost64 : kCost128;
  std::vector<long long> cost(a.items);
  std::vector<int> order(a.items);
  for (int i = 0; i < a.items; ++i) {
    const Item it = item_of(a, i);
    const Sched& sc = it.sched;
    const int tiles = sc.count(), partial = (sc.n_clean - sc.clean_full) + sc.n_noisy;
    long long c = static_cast<long long>(tiles) * (it.two_q ? cm.c2 : cm.c1) + cm.o;
    if (!it.two_q) c += static_cast<long long>(partial) * cm.p1;
    if (it.j == 0) c += static_cast<long long>(tiles) * cm.sp;
    cost[i] = c;
    order[i] = i;
  }
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return cost[x] > cost[y]; });
  std::vector<long long> load(grid, 0);
  std::vector<std::vector<int>> lists(grid);
  for (int i : order) {
    int best = 0;
    for (int c = 1; c < grid; ++c)
      if (load[c] < load[best]) best = c;
    load[best] += cost[i];
    lists[best].push_back(i);
  }
  // refinement: a bounded number of improving moves / swaps off the most loaded CTA
  if (a.items <= 8 * grid) {
    for (int iter = 0; iter < 4 * grid; ++iter) {
      int hi = 0;
      for (int c = 1; c < grid; ++c)
        if (load[c] > load[hi]) hi = c;
      long long best_max = load[hi];
      int best_lo = -1, best_a = -1, best_b = -1;  // best_b < 0: move
      for (int lo = 0; lo < grid; ++lo) {
        if (lo == hi) continue;
        for (int ia = 0; ia < static_cast<int>(lists[hi].size()); ++ia) {
          const long long ca = cost[lists[hi][ia]];
          const long long mv = std::max(load[hi] - ca, load[lo] + ca);
          if (mv < best_max) {
            best_max = mv;
            best_lo = lo, best_a = ia, best_b = -1;
          }
          for (int ib = 0; ib < static_cast<int>(lists[lo].size()); ++ib) {
            const long long d = ca - cost[lists[lo][ib]];
            if (d <= 0) continue;
            const long long sw = std::max(load[hi] - d, load[lo] + d);
            if (sw < best_max) {
              best_max = sw;
              best_lo = lo, best_a = ia, best_b = ib;
            }
          }
        }
      }
      if (best_lo < 0) break;
      const int ia = lists[hi][best_a];
      lists[hi].erase(lists[hi].begin() + best_a);
      lists[best_lo].push_back(ia);
      load[hi] -= cost[ia];
      load[best_lo] += cost[ia];
      if (best_b >= 0) {
        const int ib = lists[best_lo][best_b];
        lists[best_lo].erase(lists[best_lo].begin() + best_b);
        lists[hi].push_back(ib);
        load[best_lo] -= cost[ib];
        load[hi] += cost[ib];
      }
    }
  }
  std::unique_ptr<Plan> p(new Plan());
  int j = 0;
  for (int c = 0; c < grid; ++c) {
    std::sort(lists[c].begin(), lists[c].end(), [&](int x, int y) { return cost[x] > cost[y]; });
    p->start[c] = static_cast<uint16_t>(j);
    for (int i : lists[c]) p->item[j++] = static_cast<uint16_t>(i);
  }
  p->start[grid] = static_cast<uint16_t>(j);
  if (cache.size() >= 16) cache.erase(cache.begin());
  PlanEntry e;
  std::copy(key, key + 8, e.key);
  if (a.items <= kSmallPlanItems) {
    e.small.reset(new SmallPlan());
    std::copy(p->start, p->start + kMaxPlanCtas + 1, e.small->start);
    std::copy(p->item, p->item + kSmallPlanItems, e.small->item);
  }
  e.plan = std::move(p);
  cache.push_back(std::move(e));
  return &cache.back();
}

template <int D>
int launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
           TrainArgs a, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(train_attn_kernel<D, kMaxPlanItems>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(train_attn_kernel<D, kSmallPlanItems>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Cfg<D>::SMEM);
    if (e != cudaSuccess) return mars_host::cuda_fail(e);
    configured = true;
  }
  const int grid = std::min(a.items, mars_host::num_sms());
  static SmallPlan none;  // unused when a.planned == 0
  std::lock_guard<std::mutex> lock(plan_mutex());
  const PlanEntry* pe = plan_for(a, D, grid);
  a.planned = pe != nullptr ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(Cfg<D>::THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg<D>::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e =
      pe == nullptr           ? cudaLaunchKernelEx(&cfg, train_attn_kernel<D, kSmallPlanItems>, tq, tk, tv, to, a, none)
      : pe->small != nullptr ? cudaLaunchKernelEx(&cfg, train_attn_kernel<D, kSmallPlanItems>, tq, tk, tv, to, a, *pe->small)
                              : cudaLaunchKernelEx(&cfg, train_attn_kernel<D, kMaxPlanItems>, tq, tk, tv, to, a, *pe->plan);
  return e == cudaSuccess ? MARS_OK : mars_host::cuda_fail(e);
}

}  // namespace

extern "C" int mars_train_attn(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o, float* lse,
                               int batch, int L, int B, int Hq, int Hkv, int D, float scale, int32_t* status,
                               void* stream) {
  using mars_host::aligned16;
  MARS_HOST_CHECK(batch > 0 && L > 0 && L <= 65536 && B > 0 && Hq > 0 && Hkv > 0 && Hq % Hkv == 0,
                  MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(D == 64 || D == 128, MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(scale > 0.f && scale < INFINITY, MARS_ERR_INVALID_ARG);
  const void* ptrs[] = {q, k, v, o};
  for (const void* p : ptrs) MARS_HOST_CHECK(p != nullptr && aligned16(p), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(lse == nullptr || mars_host::aligned4(lse), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(status == nullptr || mars_host::aligned4(status), MARS_ERR_INVALID_ARG);
  const int nq = (L + kBM - 1) / kBM;
  MARS_HOST_CHECK(static_cast<long long>(batch) * Hq * 2 * nq < (1LL << 31), MARS_ERR_INVALID_ARG);
  int rc = mars_host::check_device();
  if (rc != MARS_OK) return rc;

  CUtensorMap tq, tk, tv, to;
  if (!make_map(&tq, q, D, Hq, 2 * L, batch, kBM) || !make_map(&tk, k, D, Hkv, 2 * L, batch, kBN) ||
      !make_map(&tv, v, D, Hkv, 2 * L, batch, kBN) || !make_map(&to, o, D, Hq, L, 2 * batch, 32))
    return MARS_ERR_CUDA;
  TrainArgs a;
  a.o = o;
  a.lse = lse;
  a.status = status;
  a.batch = batch;
  a.L = L;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = Hq / Hkv;
  a.scale_log2 = scale * kLog2e;
  a.nq = nq;
  a.pairs = (a.G + 1) / 2;
  a.items = 2 * nq * batch * Hkv * a.pairs;
  a.planned = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return D == 64 ? launch<64>(tq, tk, tv, to, a, s) : launch<128>(tq, tk, tv, to, a, s);
}
