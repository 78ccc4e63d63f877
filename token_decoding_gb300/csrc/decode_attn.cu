// decode_attn.cu - mars_decode_attn: the B appended [MASK] queries of one
// sliding-window decode step attend to their sequence's committed KV cache
// and causally to each other.
//
// Method: "MARS: Enabling Autoregressive Models Multi-Token Generation",
// Fig. 2 (right, sliding-window inference: B placeholders appended after the
// cursor, filled by one forward) and Eq. 2 (noisy intra-block causal case);
// the authors' MARS blog post, "Inference: a knob, not a mode switch".
//
// sm_103a design (HBM-bound: every cached K/V byte is read once).
//   * A unit is (sequence b, KV head g, chunk of Gc query heads of that group).
//     Its query rows are (position i, head) pairs, row = i * Gc + head, at most
//     128, so one K/V stream serves every head that shares the KV head (GQA).
//     The rows form the M = 128 side of tcgen05.mma; rows past Gc * B are zero.
//   * A unit is processed by a cluster of C CTAs; CTA rank c takes the unit's
//     64-key cache tiles c, c + C, c + 2C, ... (known before cache_len is read),
//     and the last rank also takes the tile of this step's B new keys (N = 16,
//     rows >= B zero).  At the end the per-row softmax states of all CTAs are
//     merged through distributed shared memory: no split-K partials reach global
//     memory.  Small units (<= 32 rows, e.g. batch 1) split each tile four ways by
//     keys over the four lane quarters and send each owning CTA its rows with one
//     bulk copy into that CTA's inbox.
//   * Inside a CTA the local tiles alternate between two streams A and B, each
//     with its own S and O in tensor memory and its own online softmax, so the
//     tensor pipe computes one stream's products while the other's softmax runs:
//       warp 0      TMA producer: Q once, the new-key tile once, then K and V
//                   cache tiles (SW128 boxes) into an NS-stage ring;
//       warp 1      TMEM owner and MMA issuer: S_x = Q K^T (SS), O_x += P_x V
//                   (TS: P is read from tensor memory);
//       warps 2..5  softmax of stream A, warps 6..9 of stream B (thread = query
//                   row = TMEM lane; warps whose 32 rows are all padding idle).
//   * Cache keys at or past cache_len are masked, and the V rows that hold them
//     in the last tile are zeroed in shared memory before P V reads them, so
//     whatever the cache holds there (even NaN) never reaches the output.
//   * Units are visited longest-cache-first (a rank computed in every CTA from
//     cache_len), so the long sequences start early and short ones fill in.
//   * Deferred-KV mode (the blog post's deferred-KV sampler: KV commitment
//     deferred into the next proposal forward, per-sample cursors, a
//     cache-validity bitmask).  A sequence carries S = 2B slots: slots 0..B-1
//     are the tokens committed by the previous step (valid below pending[b]),
//     slots B..2B-1 the new placeholders.  A slot's validity bit masks it as a
//     key and, as a query, makes its output row zero; V rows of invalid slots
//     are zeroed in shared memory.  The CTA that loads the new tile of head
//     chunk 0 also writes the valid pending K/V rows into the cache at the
//     cursor, so no separate forward or cache copy commits them.
// Every mbarrier wait is bounded; a wait that gives up sets MARS_DEV_TIMEOUT.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace {

using namespace mars;

constexpr int kTileKeys = 64;    // keys per cache tile
constexpr int kNewKeys = 16;     // N of the new-key tile (B <= 16)
constexpr int kRows = 128;       // MMA M: query rows of a unit, zero-padded
constexpr int kMaxCluster = 8;   // portable cluster size; the pull merge's state arrays are sized by it
constexpr int kWideCluster = 16; // small units (<= 32 rows) only, where the device schedules it
constexpr int kSortLimit = 256;  // sequences; above this units are visited in index order
constexpr int kThreads = 320;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P values stay below 2^8

template <int D>
struct DCfg {
  static constexpr int NB = D / 64;                     // 64-column SW128 boxes per row
  static constexpr int Q_BOX = kRows * 128;             // bytes of one Q box
  static constexpr int T_BOX = kTileKeys * 128;         // bytes of one K (or V) tile box
  static constexpr int N_BOX = kNewKeys * 128;          // bytes of one new-key box
  static constexpr int NS = D == 64 ? 8 : 5;            // ring stages
  static constexpr int Q_OFF = 0;
  static constexpr int NK_OFF = Q_OFF + NB * Q_BOX;     // new K boxes, then new V boxes
  static constexpr int NV_OFF = NK_OFF + NB * N_BOX;
  static constexpr int RING_OFF = NV_OFF + NB * N_BOX;  // stage s: K boxes then V boxes
  static constexpr int STAGE = 2 * NB * T_BOX;
  // Small-unit cluster merge (units of <= 32 rows): a row's state travels as D + 4
  // floats (acc[D], m, l, two pad), ROWB bytes.  The inbox holds one block per
  // source CTA of the rows this CTA finishes: [C][rows_per][D + 4].
  static constexpr int ROWB = (D + 4) * 4;
  static constexpr int IN_SLOTS = 32 + kMaxCluster - 1;  // >= ceil(R / C) * C for R <= 32
  static constexpr int INBOX_OFF = RING_OFF + NS * STAGE;
  static constexpr int INBOX_BYTES = IN_SLOTS * ROWB;
  // the in-CTA combine of the small-unit merge overlays the ring: 8 states x 32 rows
  // of acc, their m and l, then the outbox [32][D + 4]
  static constexpr int XCH_BYTES = 8 * 32 * D * 4 + 2 * 8 * 32 * 4 + 32 * ROWB;
  static_assert(XCH_BYTES <= NS * STAGE, "small-unit combine must fit in the ring");
  static constexpr int SMEM = INBOX_OFF + INBOX_BYTES + 1024;  // + slack to align the base to 1024
  static constexpr int TMEM_COLS = D == 64 ? 256 : 512;       // S_A | S_B | O_A | O_B
  static constexpr int O_COL = 2 * kTileKeys;
  // end-of-kernel merge state (overlays the ring): acc [2][128][D] f32, m [2][128], l [2][128],
  // then this CTA's merge weights [128][2 * kMaxCluster]
  static constexpr int MERGE_BYTES = 2 * kRows * D * 4 + 4 * kRows * 4 + kRows * 2 * kMaxCluster * 4;
  static_assert(MERGE_BYTES <= NS * STAGE, "merge state must fit in the ring");
};

struct DecodeArgs {
  const int32_t* cache_len;
  const int32_t* pending;  // deferred-KV mode: valid pending slots per sequence; nullptr otherwise
  const uint16_t* k_new;   // [batch, S, Hkv, D] (read by the fused append of pending rows)
  const uint16_t* v_new;
  uint16_t* k_cache;       // [batch, Hkv, cap, D] (written by the fused append)
  uint16_t* v_cache;
  uint16_t* o;
  int32_t* status;
  int batch, B, Hq, Hkv, cap, max_len;
  int S;             // query / new-key slots per sequence: B, or 2B in deferred-KV mode
  float scale_log2;  // scale * log2(e)
  int G;             // Hq / Hkv
  int Gc;            // query heads per unit
  int nhc;           // head chunks per KV head
  int C;             // CTAs per unit (cluster size)
  int sort_units;
  int box_rows;      // rows of a cache-tile TMA box: min(64, cap)
};

// SW128 shared-memory matrix descriptor (tcgen05 format).
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

// kSmall: the small-unit path (<= 32 rows over a cluster) is its own instantiation, so
// each launch runs only the code it needs (a single wave of CTAs, each running once,
// fetches its instructions cold).
template <int D, bool kSmall>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kc,
                  const __grid_constant__ CUtensorMap tm_vc, const __grid_constant__ CUtensorMap tm_kn,
                  const __grid_constant__ CUtensorMap tm_vn, const DecodeArgs a) {
  using C = DCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar_q, bar_new, bar_kv[C::NS], bar_kv_empty[C::NS], bar_s[2], bar_p[2], bar_o[2],
      bar_in;
  __shared__ float s_wmerge[C::IN_SLOTS];  // small-unit merge weights, [rows_per][C]
  __shared__ uint32_t tmem_slot;
  __shared__ int s_b;
  __shared__ float s_mstate[2][kRows], s_lstate[2][kRows];  // each stream's (m, l) per row (one-CTA and small units)
  __shared__ int s_len[kSortLimit];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int units_per_b = a.Hkv * a.nhc;
  const int unit_rank = blockIdx.x / a.C;
  const int crank = static_cast<int>(cluster_ctarank());

  const int R = a.Gc * a.S;            // rows loaded (row = slot i * Gc + head)
  const int act_warps = (R + 31) / 32;  // softmax warps per stream with real rows
  // Small units split over a cluster (R <= 32 rows): Q is loaded into all four
  // tensor-memory lane quarters, so each stream's S tile is split four ways by keys
  // among warps on the four SM sub-partitions (16 keys of each 64-key tile per
  // warp).  A CTA combines its 8 states of a row (2 streams x 4 quarters) and sends
  // each owning CTA its rows with one bulk copy into that CTA's inbox.
  // The small-unit instantiation compiles only its own path.  The other keeps the
  // test at run time: compiled without the small path, its register allocation ran
  // the batch-64 launch 4% slower (55.2 -> 57.4 us, measured), so it keeps both.
  const bool split4 = kSmall || (R <= 32 && a.C > 1);
  const int rows_per = (R + a.C - 1) / a.C;  // rows finished by each CTA of a small unit
  const int nrow_own = max(0, min(R, (crank + 1) * rows_per) - crank * rows_per);
  if (tid == 0) {
    mbar_init(&bar_q, 1);
    mbar_init(&bar_new, 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&bar_kv[s], 1);
      mbar_init(&bar_kv_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bar_s[x], 1);
      mbar_init(&bar_p[x], split4 ? 128 : 32 * act_warps);
      mbar_init(&bar_o[x], 1);
    }
    mbar_init(&bar_in, 1);
    fence_mbar_init();
    // small units: this CTA's inbox expects its rows from every CTA of the cluster
    if (split4) mbar_arrive_expect_tx(&bar_in, static_cast<uint32_t>(a.C * nrow_own * C::ROWB));
  }
  // matched by the wait before the first bulk copy into a peer: by then every CTA of
  // the cluster has started and armed its inbox
  if (split4) cluster_arrive_relaxed();
  if (tid == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_kc);
    tma_prefetch_desc(&tm_vc);
    tma_prefetch_desc(&tm_kn);
    tma_prefetch_desc(&tm_vn);
  }
  const uint32_t q_s = smem_u32(smem + C::Q_OFF);
  const uint32_t nk_s = smem_u32(smem + C::NK_OFF);
  const uint32_t nv_s = smem_u32(smem + C::NV_OFF);
  const uint32_t ring = smem_u32(smem + C::RING_OFF);
  // Set-up that touches no global memory runs before the wait below, beside the
  // tail of the previous kernel: zero the rows the TMA loads never write (Q rows
  // >= R, new-key rows >= S: the tail of every Q box and of every new-key box) and
  // allocate tensor memory.
  if (split4) {  // zero rows [32 j + R, 32 j + 32) of each lane quarter j
    for (int bx = 0; bx < C::NB; ++bx)
      for (int e = tid; e < 4 * (32 - R) * 8; e += kThreads) {
        const int j = e / ((32 - R) * 8), w = e % ((32 - R) * 8);
        st_shared_v4(q_s + bx * C::Q_BOX + (32 * j + R) * 128 + w * 16, 0u, 0u, 0u, 0u);
      }
  } else {
    for (int bx = 0; bx < C::NB; ++bx)
      for (int e = tid; e < (kRows - R) * 8; e += kThreads) st_shared_v4(q_s + bx * C::Q_BOX + R * 128 + e * 16, 0u, 0u, 0u, 0u);
  }
  for (int bx = 0; bx < 2 * C::NB; ++bx)  // new K boxes, then new V boxes
    for (int e = tid; e < (kNewKeys - a.S) * 8; e += kThreads)
      st_shared_v4(nk_s + bx * C::N_BOX + a.S * 128 + e * 16, 0u, 0u, 0u, 0u);
  fence_async_smem();
  if (warp == 1) tmem_alloc(&tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  // launched as a programmatic dependent: nothing global is read before the previous
  // kernel in the stream has completed
  griddep_wait();
  // The next kernel may start its set-up now, on the SMs this grid leaves free (a
  // small batch uses few); it reads nothing this kernel writes before its own wait.
  griddep_launch_dependents();

  // ---- which sequence: heavy-first rank order (stable by index) or plain order
  const int b_rank = unit_rank / units_per_b;
  const int rem = unit_rank % units_per_b;
  const int g = rem / a.nhc;
  const int hc = rem % a.nhc;
  const int h0 = g * a.G + hc * a.Gc;            // first query head of this unit
  const int heads = min(a.Gc, a.G - hc * a.Gc);  // real heads in this unit
  const bool has_new = crank == a.C - 1;
  // CTA rank c of a unit takes the unit's cache tiles c, c + C, c + 2 C, ...: local
  // tile k is global tile c + k C, which is known before cache_len is read.
  const uint32_t tile_bytes = C::NB * 128 * a.box_rows;
  auto load_tile = [&](int k, int bseq) {  // TMA loads of local cache tile k into its (free) ring stage
    const int st = k % C::NS;
    const int key0 = (crank + k * a.C) * kTileKeys;
    const uint32_t kb = ring + st * C::STAGE, vb = kb + C::NB * C::T_BOX;
    mbar_arrive_expect_tx(&bar_kv[st], 2 * tile_bytes);
    for (int c = 0; c < C::NB; ++c) {
      tma_load_4d(kb + c * C::T_BOX, &tm_kc, &bar_kv[st], 64 * c, key0, g, bseq);
      tma_load_4d(vb + c * C::T_BOX, &tm_vc, &bar_kv[st], 64 * c, key0, g, bseq);
    }
  };
  // The first loads, issued by the lanes of warp 0 side by side: lane 0 the Q tile,
  // lane 1 + k the ring stage of local cache tile k, lane NS + 1 the new-key tile
  // (each has its own barrier).  They write rows the zeroing above never touched.
  auto first_loads = [&](int bseq, int ncache_first, bool with_q) {
    if (warp != 0) return;
    if (lane == 0 && with_q) {
      mbar_arrive_expect_tx(&bar_q, C::NB * 128 * R * (split4 ? 4 : 1));
      for (int c = 0; c < C::NB; ++c)
        for (int j = 0; j < (split4 ? 4 : 1); ++j)  // split4: a copy at rows 0, 32, 64, 96
          tma_load_4d(q_s + c * C::Q_BOX + j * 32 * 128, &tm_q, &bar_q, 64 * c, h0, 0, bseq);
    } else if (lane >= 1 && lane <= ncache_first) {
      load_tile(lane - 1, bseq);
    } else if (lane == C::NS + 1 && has_new) {
      mbar_arrive_expect_tx(&bar_new, 2 * C::NB * 128 * a.S);
      for (int c = 0; c < C::NB; ++c) {
        tma_load_4d(nk_s + c * C::N_BOX, &tm_kn, &bar_new, 64 * c, g, 0, bseq);
        tma_load_4d(nv_s + c * C::N_BOX, &tm_vn, &bar_new, 64 * c, g, 0, bseq);
      }
    }
  };
  // In plain order the sequence is known at once, so Q, the new-key tile and this
  // rank's first NS cache tiles (those that start inside the cache's capacity) are
  // requested before cache_len is read: the read's latency then overlaps the loads.
  // Loaded tiles past cache_len are never used; they are waited for before exit.
  int nspec = 0;
  if (!a.sort_units) {
    while (nspec < C::NS && (crank + nspec * a.C) * kTileKeys < a.cap) ++nspec;
    first_loads(b_rank, nspec, true);
  }
  // waits for the loads issued before cache_len was read that no product will consume
  auto drain_spec = [&](int ncache_used, bool q_used) {
    if (warp != 0 || lane != 0 || a.sort_units) return;
    bool fine = true;
    if (!q_used) fine = mbar_wait(&bar_q, 0) && fine;
    for (int k = ncache_used; k < nspec; ++k) fine = mbar_wait(&bar_kv[k], 0) && fine;
    if (!fine) set_status(a.status, MARS_DEV_TIMEOUT);
  };

  if (a.sort_units) {
    for (int t = tid; t < a.batch; t += kThreads) s_len[t] = __ldg(a.cache_len + t);
    __syncthreads();
    // rank(t) = #{u : len_u > len_t, or len_u == len_t and u < t}: one thread per t,
    // every thread of a warp reading the same s_len[u] (a broadcast)
    for (int t = tid; t < a.batch; t += kThreads) {
      const int lt = s_len[t];
      int rank = 0;
      for (int u = 0; u < a.batch; ++u) {
        const int lu = s_len[u];
        rank += (lu > lt || (lu == lt && u < t)) ? 1 : 0;
      }
      if (rank == b_rank) s_b = t;
    }
    __syncthreads();
  }
  const int b = a.sort_units ? s_b : b_rank;

  const int len = a.sort_units ? s_len[b] : __ldg(a.cache_len + b);
  const bool deferred = a.pending != nullptr;
  const int pend = deferred ? __ldg(a.pending + b) : 0;
  const bool len_bad = len < 0 || len > a.max_len || pend < 0 || pend > a.B;
  if (len_bad || len + pend > a.cap) {
    // Uniform over the cluster: every CTA of the unit sees the same len and returns here.
    if (crank == 0) {
      if (tid == 0) set_status(a.status, len_bad ? MARS_DEV_LEN_RANGE : MARS_DEV_CAPACITY);
      for (int e = tid; e < heads * a.S * (D / 8); e += kThreads) {
        const int r = e / (D / 8), c = e % (D / 8);
        const int hl = r / a.S, i = r % a.S;
        *reinterpret_cast<uint4*>(a.o + ((static_cast<size_t>(b) * a.S + i) * a.Hq + h0 + hl) * D + 8 * c) =
            make_uint4(0, 0, 0, 0);
      }
    }
    drain_spec(0, false);  // the early loads land before the CTA exits
    if (warp == 0 && lane == 0 && has_new && !a.sort_units && !mbar_wait(&bar_new, 0))
      set_status(a.status, MARS_DEV_TIMEOUT);
    __syncthreads();  // tensor memory was allocated before the wait: free it (no product was issued)
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem_slot, C::TMEM_COLS);
    }
    return;
  }
  // slot validity bitmask: every slot, or (deferred) the pending slots below pend and all placeholders
  const uint32_t vmask = deferred ? ((1u << pend) - 1u) | (((1u << a.B) - 1u) << a.B) : (1u << a.S) - 1u;
  const int nct = (len + kTileKeys - 1) / kTileKeys;  // cache tiles of the unit
  const int ncache = nct > crank ? (nct - crank + a.C - 1) / a.C : 0;  // local cache tiles
  const int ntiles = ncache + (has_new ? 1 : 0);  // local tile k: cache tile crank + k C, then the new tile
  if (a.sort_units && ntiles > 0) first_loads(b, min(ncache, C::NS), true);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  bool ok = true;

  if (warp == 0) {
    // ================= TMA producer: the tiles past the first NS, each into a freed stage
    // (everything it loads is consumed, or waited for, before the CTA exits)
    if (lane == 0) {
      for (int k = C::NS; k < ncache; ++k) {
        if (!mbar_wait(&bar_kv_empty[k % C::NS], ((k / C::NS) - 1) & 1)) {
          set_status(a.status, MARS_DEV_TIMEOUT);
          break;
        }
        load_tile(k, b);
      }
    }
    drain_spec(ncache, ntiles > 0);
    __syncwarp();
    if (deferred && has_new && hc == 0) {
      // Commit the valid pending rows of KV head g at the cursor.  Other CTAs of
      // this sequence may load these cache rows inside their last tile at the same
      // time; they mask them (keys at or past cache_len), so either value is fine.
      constexpr int vpr = D / 8;  // 16-byte vectors per row
      for (int e = lane; e < pend * vpr; e += 32) {
        const int i = e / vpr, c = e % vpr;
        const size_t src = ((static_cast<size_t>(b) * a.S + i) * a.Hkv + g) * D + 8 * c;
        const size_t dst = ((static_cast<size_t>(b) * a.Hkv + g) * a.cap + len + i) * D + 8 * c;
        *reinterpret_cast<uint4*>(a.k_cache + dst) = *reinterpret_cast<const uint4*>(a.k_new + src);
        *reinterpret_cast<uint4*>(a.v_cache + dst) = *reinterpret_cast<const uint4*>(a.v_new + src);
      }
    }
  } else if (warp == 1) {
    // ================= MMA issuer.  The whole warp runs the schedule, so the
    // descriptors stay warp-uniform; one elected lane issues the tcgen05
    // operations and their commits (a commit tracks its own thread's MMAs).
    if (ntiles > 0) {
      const bool leader = elect_one();
      constexpr uint32_t id_qk = idesc_bf16(kRows, kTileKeys, false);
      constexpr uint32_t id_qn = idesc_bf16(kRows, kNewKeys, false);
      constexpr uint32_t id_pv = idesc_bf16(kRows, D, true);
      const uint64_t desc_q = smem_desc(q_s, 16, 1024);
      const uint64_t desc_nk = smem_desc(nk_s, 16, 1024);
      const uint64_t desc_nv = smem_desc(nv_s, C::N_BOX, 1024);
      const uint64_t desc_k = smem_desc(ring, 16, 1024);
      const uint64_t desc_v = smem_desc(ring + C::NB * C::T_BOX, C::T_BOX, 1024);
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_q, 0));
      // Descriptor start addresses are in 16-byte units, so stepping by `bytes` adds bytes >> 4.
      auto issue_qk = [&](int k) {
        const uint32_t d_tmem = tmem + (k & 1) * kTileKeys;
        const bool cache_tile = k < ncache;
        const int st = k % C::NS;
        ok = ok && __all_sync(0xffffffffu, cache_tile ? mbar_wait(&bar_kv[st], (k / C::NS) & 1) : mbar_wait(&bar_new, 0));
        if (!ok) return;
        tc_fence_after();
        if (leader) {
          if (cache_tile) {
            const uint64_t kb = desc_k + ((st * C::STAGE) >> 4);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              tc_mma_ss(d_tmem, desc_q + (((ks >> 2) * C::Q_BOX + (ks & 3) * 32) >> 4),
                        kb + (((ks >> 2) * C::T_BOX + (ks & 3) * 32) >> 4), id_qk, ks > 0 ? 1u : 0u);
          } else {
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              tc_mma_ss(d_tmem, desc_q + (((ks >> 2) * C::Q_BOX + (ks & 3) * 32) >> 4),
                        desc_nk + (((ks >> 2) * C::N_BOX + (ks & 3) * 32) >> 4), id_qn, ks > 0 ? 1u : 0u);
          }
          tc_commit(&bar_s[k & 1]);
        }
        __syncwarp();
      };
      auto issue_pv = [&](int k) {
        const int x = k & 1;
        const bool cache_tile = k < ncache;
        const int st = k % C::NS;
        // K and V of the tile arrived before its S product was issued
        ok = ok && __all_sync(0xffffffffu, mbar_wait(&bar_p[x], (k >> 1) & 1));
        if (!ok) return;
        tc_fence_after();
        const uint32_t p_tmem = tmem + x * kTileKeys;  // P as bf16 pairs in the first 32 columns of S_x
        const uint32_t o_tmem = tmem + C::O_COL + x * D;
        const bool first = k < 2;
        if (leader) {
          if (cache_tile) {
            const uint64_t vb = desc_v + ((st * C::STAGE) >> 4);
#pragma unroll
            for (int ks = 0; ks < kTileKeys / 16; ++ks)
              tc_mma_ts(o_tmem, p_tmem + ks * 8, vb + ((ks * 16 * 128) >> 4), id_pv, (!first || ks > 0) ? 1u : 0u);
            tc_commit(&bar_kv_empty[st]);
          } else {
            tc_mma_ts(o_tmem, p_tmem, desc_nv, id_pv, first ? 0u : 1u);
          }
          if (k + 2 >= ntiles) tc_commit(&bar_o[x]);  // the stream's last product
        }
        __syncwarp();
      };
      if (ok) issue_qk(0);
      if (ok && ntiles > 1) issue_qk(1);
      // S_x(k+2) is issued after O_x += P_x(k) V(k): when S_x(k+2) is complete, so is
      // every earlier product of stream x, which the softmax relies on to rescale O_x.
      for (int k = 0; ok && k < ntiles; ++k) {
        issue_pv(k);
        if (ok && k + 2 < ntiles) issue_qk(k + 2);
      }
      if (!ok && leader) set_status(a.status, MARS_DEV_TIMEOUT);
    }
    __syncwarp();
  } else if (split4) {
    // ================= small unit: the softmax warp of stream x in lane quarter q
    // (warps 2..5: A, 6..9: B) takes keys [16 q, 16 q + 16) of each of the stream's
    // tiles for every row (thread = row, the same rows in every quarter).  Its P
    // goes to columns [8 q, 8 q + 8) of the tile's P and zeros to the other 24, so
    // the PV product of a quarter's lanes sums its own keys only.
    const int x = (warp - 2) >> 2;
    const int q = warp & 3;
    const int r = lane;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t s_col = tmem + lane_addr + x * kTileKeys;
    const uint32_t o_col = tmem + lane_addr + C::O_COL + x * D;
    const int slot = r / a.Gc;
    const bool row_valid = r < R && slot < a.S && ((vmask >> slot) & 1u);
    const uint32_t new_vis = row_valid ? vmask & ((2u << slot) - 1u) : 0u;
    float m_used = -INFINITY, l = 0.f;
    int nmine = 0;
    for (int k = x; k < ntiles; k += 2, ++nmine) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_s[x], nmine & 1));
      if (!ok) break;
      tc_fence_after();
      const bool is_new = k >= ncache;
      const int tile0 = (crank + k * a.C) * kTileKeys;  // first key of the (cache) tile
      uint32_t sv[16];
      tmem_ld16(s_col + 16 * q, sv);
      tc_wait_ld();
      if (is_new) {
        // the new-key tile has kNewKeys = 16 keys, all in quarter 0's slice
#pragma unroll
        for (int c = 0; c < 16; ++c) sv[c] = (q == 0 && ((new_vis >> c) & 1u)) ? sv[c] : 0xFF800000u;
      } else {
        const int vlast = row_valid ? len - 1 - tile0 - 16 * q : -1;  // last visible key of the slice
        if (vlast < 15) {
#pragma unroll
          for (int c = 0; c < 16; ++c) sv[c] = c <= vlast ? sv[c] : 0xFF800000u;
        }
      }
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int c = 0; c < 16; c += 2) {
        mx0 = fmaxf(mx0, __uint_as_float(sv[c]));
        mx1 = fmaxf(mx1, __uint_as_float(sv[c + 1]));
      }
      const float tile_max = fmaxf(mx0, mx1) * a.scale_log2;
      float alpha = 1.f;
      const bool grow = tile_max > m_used + kRescaleThreshold;
      if (grow) {
        alpha = fast_exp2(m_used - tile_max);  // 0 when m_used is -inf
        m_used = tile_max;
      }
      if (nmine > 0 && __any_sync(0xffffffffu, grow)) {
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
      const float neg_mu = m_used == -INFINITY ? 0.f : -m_used;
      float sum0 = 0.f, sum1 = 0.f;
      uint32_t pw[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float p0 = fast_exp2(fmaf(__uint_as_float(sv[2 * e]), a.scale_log2, neg_mu));
        const float p1 = fast_exp2(fmaf(__uint_as_float(sv[2 * e + 1]), a.scale_log2, neg_mu));
        sum0 += p0;
        sum1 += p1;
        pw[e] = pack_bf16x2(p0, p1);
      }
      uint32_t plo[16], phi[16];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        plo[e] = q == 0 ? pw[e] : 0u;
        plo[8 + e] = q == 1 ? pw[e] : 0u;
        phi[e] = q == 2 ? pw[e] : 0u;
        phi[8 + e] = q == 3 ? pw[e] : 0u;
      }
      tmem_st16(s_col, plo);
      tmem_st16(s_col + 16, phi);
      l = l * alpha + (sum0 + sum1);
      // V rows that P = 0 meets must be finite: invalid pending slots of the new tile
      // (deferred mode) and keys at or past cache_len in the last cache tile
      if (is_new && deferred && pend < a.B) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_new, 0));
        if (!ok) break;
        const int per_box = (a.B - pend) * 8;
        for (int e = q * 32 + lane; e < C::NB * per_box; e += 128) {
          const int bx = e / per_box, w = e % per_box;
          st_shared_v4(nv_s + bx * C::N_BOX + pend * 128 + w * 16, 0u, 0u, 0u, 0u);
        }
        fence_async_smem();
      }
      if (!is_new && len - tile0 < kTileKeys) {
        const int st = k % C::NS;
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_kv[st], (k / C::NS) & 1));
        if (!ok) break;
        const int z0 = len - tile0;
        const int per_box = (kTileKeys - z0) * 8;
        const uint32_t vb = ring + st * C::STAGE + C::NB * C::T_BOX;
        for (int e = q * 32 + lane; e < C::NB * per_box; e += 128) {
          const int bx = e / per_box, w = e % per_box;
          st_shared_v4(vb + bx * C::T_BOX + z0 * 128 + w * 16, 0u, 0u, 0u, 0u);
        }
        fence_async_smem();
      }
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(&bar_p[x]);
    }
    if (ok && nmine > 0) ok = __all_sync(0xffffffffu, mbar_wait(&bar_o[x], 0));
    if (!ok && lane == 0) set_status(a.status, MARS_DEV_TIMEOUT);
    const bool have = ok && nmine > 0;
    // ---- combine this CTA's 8 states of each row (stream x, lane quarter q), in two
    // levels.  The warps of streams A and B in quarter q reach the same tensor-memory
    // lanes, so each first merges the two streams' O of its rows from tensor memory,
    // warp (x, q) columns [x D / 2, (x + 1) D / 2), with weights from the exchanged
    // (m, l), and writes the quarter's state to shared memory; then warp w = 4 x + q
    // merges columns [w D / 8, (w + 1) D / 8) of the four quarter states of every row
    // into the outbox [32][D + 4]; the warp of slice 0 adds the row's (m, l).
    const int wst = x * 4 + q;
    // each stream's (m, l) of the rows, exchanged outside the ring (the other stream's
    // products may still read the ring until the barrier below)
    s_mstate[x][q * 32 + r] = have ? m_used : -INFINITY;
    s_lstate[x][q * 32 + r] = have ? l : 0.f;
    named_bar_sync(1, 256);  // every product of both streams is complete: the ring is free
    tc_fence_after();
    float* xo = reinterpret_cast<float*>(smem + C::RING_OFF);  // [4][32][D] used, 16-byte units XOR (row & 7)
    float* xm = xo + 8 * 32 * D;                               // [4][32] used: the quarters' m
    float* xl = xm + 8 * 32;                                   // [4][32] used: the quarters' l
    float* outbox = xl + 8 * 32;                               // [32][D + 4]
    {
      const float mx_ = s_mstate[x][q * 32 + r], my = s_mstate[1 - x][q * 32 + r];
      const float mq = fmaxf(mx_, my);
      // weights of this stream (x) and the other (y); a stream without keys weighs 0
      // and its accumulator (never written when it had no tile) is not read into the sum
      const float wx = mx_ == -INFINITY ? 0.f : fast_exp2(mx_ - mq);
      const float wy = my == -INFINITY ? 0.f : fast_exp2(my - mq);
      const uint32_t ox_col = o_col, oy_col = tmem + lane_addr + C::O_COL + (1 - x) * D;
      float4* dst = reinterpret_cast<float4*>(xo + (q * 32 + r) * D);
#pragma unroll 1
      for (int c = x * (D / 2); c < (x + 1) * (D / 2); c += 32) {
        uint32_t vx[32], vy[32];
        tmem_ld32(ox_col + c, vx);
        tmem_ld32(oy_col + c, vy);
        tc_wait_ld();
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float4 v;
          v.x = (wx > 0.f ? wx * __uint_as_float(vx[4 * e]) : 0.f) + (wy > 0.f ? wy * __uint_as_float(vy[4 * e]) : 0.f);
          v.y = (wx > 0.f ? wx * __uint_as_float(vx[4 * e + 1]) : 0.f) +
                (wy > 0.f ? wy * __uint_as_float(vy[4 * e + 1]) : 0.f);
          v.z = (wx > 0.f ? wx * __uint_as_float(vx[4 * e + 2]) : 0.f) +
                (wy > 0.f ? wy * __uint_as_float(vy[4 * e + 2]) : 0.f);
          v.w = (wx > 0.f ? wx * __uint_as_float(vx[4 * e + 3]) : 0.f) +
                (wy > 0.f ? wy * __uint_as_float(vy[4 * e + 3]) : 0.f);
          dst[((c >> 2) + e) ^ (r & 7)] = v;
        }
      }
      if (x == 0) {  // the quarter's state: max mq, sum of the weighted l
        xm[q * 32 + r] = mq;
        xl[q * 32 + r] = wx * s_lstate[0][q * 32 + r] + wy * s_lstate[1][q * 32 + r];
      }
    }
    named_bar_sync(1, 256);
    if (r < R) {
      float ws[4];
      float mx = -INFINITY;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        ws[t] = xm[t * 32 + r];
        mx = fmaxf(mx, ws[t]);
      }
      float lsum = 0.f;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        ws[t] = ws[t] == -INFINITY ? 0.f : fast_exp2(ws[t] - mx);  // states without keys weigh 0
        lsum += ws[t] * xl[t * 32 + r];
      }
      const float4* x4 = reinterpret_cast<const float4*>(xo);
      float4* orow = reinterpret_cast<float4*>(outbox + r * (D + 4));
#pragma unroll
      for (int j = 0; j < D / 32; ++j) {
        const int c4 = wst * (D / 32) + j;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float4 v = x4[(t * 32 + r) * (D / 4) + (c4 ^ (r & 7))];
          acc.x += ws[t] * v.x;
          acc.y += ws[t] * v.y;
          acc.z += ws[t] * v.z;
          acc.w += ws[t] * v.w;
        }
        orow[c4] = acc;
      }
      if (wst == 0) orow[D / 4] = make_float4(mx, lsum, 0.f, 0.f);
    }
    fence_async_smem();  // the bulk copies (async proxy) read the outbox
    named_bar_sync(1, 256);
  } else {
    // ================= softmax of stream x (warps 2..5: A, 6..9: B)
    const int x = (warp - 2) >> 2;
    const int quad = warp & 3;  // TMEM lane quarter this warp may access
    const int r = quad * 32 + lane;
    const bool active = quad < act_warps;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_col = tmem + lane_addr + x * kTileKeys;
    const uint32_t o_col = tmem + lane_addr + C::O_COL + x * D;
    const int slot = r / a.Gc;  // query slot i of this row (rows >= R are padding)
    // A valid query slot sees the valid new keys up to itself; padding rows and
    // invalid slots see nothing (their outputs are zero or never written).
    const bool row_valid = slot < a.S && ((vmask >> slot) & 1u);
    const uint32_t new_vis = row_valid ? vmask & ((2u << slot) - 1u) : 0u;
    float m_used = -INFINITY, l = 0.f;
    int nmine = 0;
    if (active) {
      for (int k = x; k < ntiles; k += 2, ++nmine) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_s[x], nmine & 1));
        if (!ok) break;
        tc_fence_after();
        // last visible column of this tile for this row
        const bool is_new = k >= ncache;
        const int key0 = (crank + k * a.C) * kTileKeys;
        const int vlast = row_valid ? len - 1 - key0 : -1;
        uint32_t s[kTileKeys];
        tmem_ld32(s_col, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_ld32(s_col + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tc_wait_ld();
        if (is_new) {
#pragma unroll
          for (int c = 0; c < kTileKeys; ++c)
            s[c] = (c < kNewKeys && ((new_vis >> c) & 1u)) ? s[c] : 0xFF800000u;  // -inf
        } else if (vlast < kTileKeys - 1) {
#pragma unroll
          for (int c = 0; c < kTileKeys; ++c) s[c] = c <= vlast ? s[c] : 0xFF800000u;
        }
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int c = 0; c < kTileKeys; c += 2) {
          mx0 = fmaxf(mx0, __uint_as_float(s[c]));
          mx1 = fmaxf(mx1, __uint_as_float(s[c + 1]));
        }
        const float tile_max = fmaxf(mx0, mx1) * a.scale_log2;
        // lazy rescale: keep the old reference max unless the new one is 2^8 larger
        float alpha = 1.f;
        const bool grow = tile_max > m_used + kRescaleThreshold;
        if (grow) {
          alpha = fast_exp2(m_used - tile_max);  // 0 when m_used is -inf
          m_used = tile_max;
        }
        if (nmine > 0 && __any_sync(0xffffffffu, grow)) {
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
        const float neg_mu = m_used == -INFINITY ? 0.f : -m_used;
        float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
        for (int c = 0; c < kTileKeys; c += 32) {
          uint32_t pw[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float p0 = fast_exp2(fmaf(__uint_as_float(s[c + 2 * e]), a.scale_log2, neg_mu));
            const float p1 = fast_exp2(fmaf(__uint_as_float(s[c + 2 * e + 1]), a.scale_log2, neg_mu));
            sum0 += p0;
            sum1 += p1;
            pw[e] = pack_bf16x2(p0, p1);
          }
          tmem_st16(s_col + (c >> 1), pw);
        }
        l = l * alpha + (sum0 + sum1);
        // Invalid pending slots of the new tile may hold anything (even NaN): zero
        // their V rows so that P = 0 meets finite values.
        if (is_new && deferred && pend < a.B) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bar_new, 0));
          if (!ok) break;
          const int per_box = (a.B - pend) * 8;  // 16-byte chunks of rows pend .. B-1
          for (int e = quad * 32 + lane; e < C::NB * per_box; e += 32 * act_warps) {
            const int bx = e / per_box, w = e % per_box;
            st_shared_v4(nv_s + bx * C::N_BOX + pend * 128 + w * 16, 0u, 0u, 0u, 0u);
          }
          fence_async_smem();
        }
        // The last cache tile can hold keys at or past cache_len: zero those V rows
        // (whole 128-byte rows of every box) so that P = 0 meets finite values.
        if (!is_new && len - key0 < kTileKeys) {
          const int st = k % C::NS;
          ok = __all_sync(0xffffffffu, mbar_wait(&bar_kv[st], (k / C::NS) & 1));
          if (!ok) break;
          const int z0 = len - key0;
          const int per_box = (kTileKeys - z0) * 8;  // 16-byte chunks
          const uint32_t vb = ring + st * C::STAGE + C::NB * C::T_BOX;
          for (int e = quad * 32 + lane; e < C::NB * per_box; e += 32 * act_warps) {
            const int bx = e / per_box, w = e % per_box;
            st_shared_v4(vb + bx * C::T_BOX + z0 * 128 + w * 16, 0u, 0u, 0u, 0u);
          }
          fence_async_smem();
        }
        tc_wait_st();
        tc_fence_before();
        mbar_arrive(&bar_p[x]);
      }
      if (ok && nmine > 0) ok = __all_sync(0xffffffffu, mbar_wait(&bar_o[x], 0));
      if (!ok && lane == 0) set_status(a.status, MARS_DEV_TIMEOUT);
    }
    const bool have = ok && nmine > 0;
    if (a.C == 1) {
      // ---- one CTA per unit: combine the two streams of each row straight from
      // tensor memory.  Thread (stream x, row r) writes columns [x D/2, (x+1) D/2)
      // of the row, reading both streams' O there.
      if (active) {
        s_mstate[x][r] = have ? m_used : -INFINITY;
        s_lstate[x][r] = have ? l : 0.f;
      }
      named_bar_sync(1, 256);
      tc_fence_after();
      if (active) {
        const float m0 = s_mstate[0][r], m1 = s_mstate[1][r];
        const float mmax = fmaxf(m0, m1);
        float w0 = m0 == -INFINITY ? 0.f : fast_exp2(m0 - mmax);
        float w1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - mmax);
        const float lsum = w0 * s_lstate[0][r] + w1 * s_lstate[1][r];
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;  // 0: a row that sees no key (padding, invalid slot)
        w0 *= inv;
        w1 *= inv;
        const int i = r / a.Gc, hl = r % a.Gc;
        const bool store = r < R && hl < heads;
        const uint32_t oa = tmem + lane_addr + C::O_COL + x * (D / 2);  // stream A's O, this half
        const uint32_t ob = oa + D;                                      // stream B's O, this half
        uint4* dst = reinterpret_cast<uint4*>(a.o + ((static_cast<size_t>(b) * a.S + i) * a.Hq + h0 + hl) * D +
                                              x * (D / 2));
#pragma unroll 1
        for (int c = 0; c < D / 2; c += 32) {
          uint32_t va[32], vb[32];
          tmem_ld32(oa + c, va);
          tmem_ld32(ob + c, vb);
          tc_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            // a stream without tiles never wrote its O: its weight is 0 and its columns are not read
            const float f0 = (w0 != 0.f ? w0 * __uint_as_float(va[2 * e]) : 0.f) +
                             (w1 != 0.f ? w1 * __uint_as_float(vb[2 * e]) : 0.f);
            const float f1 = (w0 != 0.f ? w0 * __uint_as_float(va[2 * e + 1]) : 0.f) +
                             (w1 != 0.f ? w1 * __uint_as_float(vb[2 * e + 1]) : 0.f);
            pk[e] = pack_bf16x2(f0, f1);
          }
          if (store) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[(c >> 3) + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      }
    } else {
      // Both streams' products are complete once every softmax warp is past its
      // wait above, so the ring (every loaded tile consumed) can hold the merge state.
      named_bar_sync(1, 256);
      tc_fence_after();
      float* acc_s = reinterpret_cast<float*>(smem + C::RING_OFF);  // [2][128][D], 16-byte units XOR (row & 7)
      float* m_s = acc_s + 2 * kRows * D;                           // [2][128]
      float* l_s = m_s + 2 * kRows;                                 // [2][128]
      if (active) {
        float4* dst = reinterpret_cast<float4*>(acc_s + (x * kRows + r) * D);
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          uint32_t ov[32];
          tmem_ld32(o_col + c, ov);
          tc_wait_ld();
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 v = have ? make_float4(__uint_as_float(ov[4 * e]), __uint_as_float(ov[4 * e + 1]),
                                                __uint_as_float(ov[4 * e + 2]), __uint_as_float(ov[4 * e + 3]))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            dst[((c >> 2) + e) ^ (r & 7)] = v;
          }
        }
        m_s[x * kRows + r] = have ? m_used : -INFINITY;
        l_s[x * kRows + r] = have ? l : 0.f;
      }
    }
  }

  // ---- merge the 2 * C states of every row through distributed shared memory.
  // This CTA finishes rows [r_lo, r_hi): first one weight per (row, state),
  // w = 2^(m - max m) / sum_states(2^(m - max m) l), then O = sum w acc.
  tc_fence_before();
  if (split4) {
    // Each owning CTA (rows [o rows_per, (o + 1) rows_per)) receives this CTA's combined
    // rows as one bulk copy into block `crank` of its inbox, completing on its bar_in.
    cluster_wait();  // every CTA of the cluster has started and armed its inbox
    // Lane o of warp 2 sends owner o its rows, so the copies are issued side by side
    // (C <= 32); each lane later waits for its own copy's reads.
    if (warp == 2 && lane < a.C) {
      const uint32_t ob = smem_u32(smem + C::RING_OFF) + 8 * 32 * D * 4 + 2 * 8 * 32 * 4;
      const uint32_t inbox = smem_u32(smem + C::INBOX_OFF) + crank * rows_per * C::ROWB;
      const int o = lane;
      const int n_o = min(rows_per, R - o * rows_per);
      if (n_o > 0)
        bulk_s2s_cluster(dsmem_map(inbox, o), ob + o * rows_per * C::ROWB, n_o * C::ROWB,
                         dsmem_map(smem_u32(&bar_in), o));
      bulk_commit_group();
    }
    // Finish the owned rows from the inbox: one weight per (row, source),
    // w = 2^(m - max m) / sum(2^(m - max m) l), then O = sum w acc.
    const bool got = nrow_own == 0 || __syncthreads_and(mbar_wait(&bar_in, 0));
    if (!got) {
      if (tid == 0) set_status(a.status, MARS_DEV_TIMEOUT);
    } else if (nrow_own > 0) {
      const float* in = reinterpret_cast<const float*>(smem + C::INBOX_OFF);  // [C][rows_per][D + 4]
      for (int t0 = 0; t0 < nrow_own * a.C; t0 += kThreads) {  // uniform trip count: every lane shuffles
        const int t = t0 + tid;  // (row rr, source c) = (t / C, t % C)
        const bool valid = t < nrow_own * a.C;
        const float* st = in + ((t % a.C) * rows_per + t / a.C) * (D + 4);
        const float m = valid ? st[D] : -INFINITY, l = valid ? st[D + 1] : 0.f;
        float mmax = m;
        for (int o = a.C >> 1; o > 0; o >>= 1) mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, o));
        const float w = m == -INFINITY ? 0.f : fast_exp2(m - mmax);
        float lsum = w * l;
        for (int o = a.C >> 1; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
        if (valid) s_wmerge[t] = lsum > 0.f ? w / lsum : 0.f;  // 0: a row that sees no key (invalid slot)
      }
      __syncthreads();
      for (int e = tid; e < nrow_own * (D / 4); e += kThreads) {
        const int rr = e / (D / 4), d4 = e % (D / 4);
        const int r = crank * rows_per + rr;
        const int i = r / a.Gc, hl = r % a.Gc;
        if (hl >= heads) continue;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int c = 0; c < kWideCluster; ++c) {  // unrolled: the sources' loads issue together
          if (c < a.C) {
            const float w = s_wmerge[rr * a.C + c];
            const float4 v = reinterpret_cast<const float4*>(in + (c * rows_per + rr) * (D + 4))[d4];
            o.x += w * v.x;
            o.y += w * v.y;
            o.z += w * v.z;
            o.w += w * v.w;
          }
        }
        uint16_t* dst = a.o + ((static_cast<size_t>(b) * a.S + i) * a.Hq + h0 + hl) * D + 4 * d4;
        *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(o.x, o.y), pack_bf16x2(o.z, o.w));
      }
    }
    if (warp == 2 && lane < a.C) bulk_wait_read_all();  // the outbox has been read: this CTA may exit
    __syncthreads();  // every tensor-memory read of the epilogue is done
  } else if (a.C > 1) {
    cluster_sync();
    {
      const float* acc_s = reinterpret_cast<const float*>(smem + C::RING_OFF);
      const float* m_s = acc_s + 2 * kRows * D;
      const float* l_s = m_s + 2 * kRows;
      float* w_s = const_cast<float*>(l_s) + 2 * kRows;  // [rows_per][2 * kMaxCluster], this CTA's own
      const uint32_t acc_l = smem_u32(acc_s), m_l = smem_u32(m_s), l_l = smem_u32(l_s);
      const int rows_per = (R + a.C - 1) / a.C;
      const int r_lo = crank * rows_per, r_hi = min(R, r_lo + rows_per);
      const int ns = 2 * a.C;  // states per row: a power of two <= 16, so a row's states are aligned lanes
      // One thread per (row, state): every state's (m, l) is requested at once, then
      // the row's max and weighted sum are reduced with shuffles among its ns lanes.
      const int nrow = r_hi - r_lo;
      for (int t0 = 0; t0 < nrow * ns; t0 += kThreads) {  // uniform trip count: every lane shuffles
        const int t = t0 + tid;
        const bool valid = t < nrow * ns;
        const int r = r_lo + t / ns, q = t % ns;
        float m = -INFINITY, l = 0.f;
        if (valid) {
          m = dsmem_ld_f32(dsmem_map(m_l + 4 * ((q & 1) * kRows + r), q >> 1));
          l = dsmem_ld_f32(dsmem_map(l_l + 4 * ((q & 1) * kRows + r), q >> 1));
        }
        float mmax = m;
        for (int o = ns >> 1; o > 0; o >>= 1) mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, o));
        const float w = m == -INFINITY ? 0.f : fast_exp2(m - mmax);
        float lsum = w * l;
        for (int o = ns >> 1; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;  // 0: a row that sees no key (invalid slot)
        if (valid) w_s[(r - r_lo) * 2 * kMaxCluster + q] = w * inv;
      }
      __syncthreads();
      for (int e = tid; e < (r_hi - r_lo) * (D / 4); e += kThreads) {
        const int r = r_lo + e / (D / 4);
        const int d4 = e % (D / 4);
        const int i = r / a.Gc, hl = r % a.Gc;
        if (hl >= heads) continue;
        const float* w = w_s + (r - r_lo) * 2 * kMaxCluster;
        const uint32_t off = acc_l + 4 * (r * D + 4 * (d4 ^ (r & 7)));
        float4 v[2 * kMaxCluster];
#pragma unroll
        for (int q = 0; q < 2 * kMaxCluster; ++q)
          if (q < ns) v[q] = dsmem_ld_f32x4(dsmem_map(off + 4 * (q & 1) * kRows * D, q >> 1));
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 2 * kMaxCluster; ++q) {
          if (q < ns) {
            o.x += w[q] * v[q].x;
            o.y += w[q] * v[q].y;
            o.z += w[q] * v[q].z;
            o.w += w[q] * v[q].w;
          }
        }
        uint16_t* dst = a.o + ((static_cast<size_t>(b) * a.S + i) * a.Hq + h0 + hl) * D + 4 * d4;
        *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(o.x, o.y), pack_bf16x2(o.z, o.w));
      }
    }
    cluster_sync();  // keep this CTA's shared memory alive until every peer has read it
  } else {
    __syncthreads();  // every tensor-memory read of the epilogue is done
  }
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

// A contiguous bf16 tensor with dims d[0] (innermost, = D) .. d[3], loaded in
// SW128 boxes of 64 x box1 x box2 x 1 elements.
bool make_map(CUtensorMap* m, const void* ptr, const long long (&d)[4], int box1, int box2) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d[0]), static_cast<cuuint64_t>(d[1]),
                              static_cast<cuuint64_t>(d[2]), static_cast<cuuint64_t>(d[3])};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d[0]) * 2, static_cast<cuuint64_t>(d[0] * d[1]) * 2,
                                 static_cast<cuuint64_t>(d[0] * d[1] * d[2]) * 2};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box1), static_cast<cuuint32_t>(box2), 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Maps {
  CUtensorMap q, kc, vc, kn, vn;
};

template <int D, bool kSmall>
int launch(const Maps& mp, DecodeArgs a, int units, cudaStream_t stream) {
  auto kern = decode_kernel<D, kSmall>;
  static bool configured = false;  // per instantiation; the attribute is process-wide
  static bool wide_ok = false;     // 16-CTA clusters (a non-portable size) can be scheduled
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DCfg<D>::SMEM);
    if (e != cudaSuccess) return mars_host::cuda_fail(e);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
      cudaLaunchConfig_t q = {};
      q.gridDim = dim3(kWideCluster, 1, 1);
      q.blockDim = dim3(kThreads, 1, 1);
      q.dynamicSmemBytes = DCfg<D>::SMEM;
      cudaLaunchAttribute qa[1];
      qa[0].id = cudaLaunchAttributeClusterDimension;
      qa[0].val.clusterDim.x = kWideCluster;
      qa[0].val.clusterDim.y = 1;
      qa[0].val.clusterDim.z = 1;
      q.attrs = qa;
      q.numAttrs = 1;
      int n = 0;
      wide_ok = cudaOccupancyMaxActiveClusters(&n, kern, &q) == cudaSuccess && n >= 4;
    }
    cudaGetLastError();  // a refused query leaves no sticky error behind
    configured = true;
  }
  if (a.C == kWideCluster && !wide_ok) a.C = kMaxCluster;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(units * a.C, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = DCfg<D>::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, mp.q, mp.kc, mp.vc, mp.kn, mp.vn, a);
  if (e != cudaSuccess) return mars_host::cuda_fail(e);
  return MARS_OK;
}

inline int ceil_div(long long x, long long y) { return static_cast<int>((x + y - 1) / y); }
inline int pow2_ceil(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

// Shared host path of both entry points: pending == nullptr is the plain step
// (S = B slots), otherwise the deferred-KV step (S = 2B slots).
int decode_impl(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new, const uint16_t* k_cache,
                const uint16_t* v_cache, uint16_t* k_cache_w, uint16_t* v_cache_w, const int32_t* cache_len,
                const int32_t* pending, int batch, int B, int Hq, int Hkv, int D, int cap, int max_len, float scale,
                uint16_t* o, int32_t* status, cudaStream_t stream) {
  using mars_host::aligned16;
  const int S = pending != nullptr ? 2 * B : B;
  MARS_HOST_CHECK(batch > 0 && B >= 1 && S <= kNewKeys && Hq > 0 && Hkv > 0 && Hq % Hkv == 0, MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(D == 64 || D == 128, MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(cap > 0 && max_len >= 0 && max_len <= cap, MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(scale > 0.f && scale < INFINITY, MARS_ERR_INVALID_ARG);
  const void* ptrs[] = {q, k_new, v_new, k_cache, v_cache, o};
  for (const void* p : ptrs) MARS_HOST_CHECK(p != nullptr && aligned16(p), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(cache_len != nullptr && mars_host::aligned4(cache_len), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(pending == nullptr || mars_host::aligned4(pending), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(status == nullptr || mars_host::aligned4(status), MARS_ERR_INVALID_ARG);
  int rc = mars_host::check_device();
  if (rc != MARS_OK) return rc;

  DecodeArgs a;
  a.cache_len = cache_len;
  a.pending = pending;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_cache = k_cache_w;
  a.v_cache = v_cache_w;
  a.o = o;
  a.status = status;
  a.batch = batch;
  a.B = B;
  a.S = S;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.cap = cap;
  a.max_len = max_len;
  a.scale_log2 = scale * kLog2e;
  a.G = Hq / Hkv;
  // Heads per unit: as many as fit in the 128 rows of one MMA tile.
  a.Gc = std::min(a.G, kRows / S);
  a.nhc = ceil_div(a.G, a.Gc);
  const long long units = static_cast<long long>(batch) * Hkv * a.nhc;
  MARS_HOST_CHECK(units * kMaxCluster < (1LL << 31), MARS_ERR_INVALID_ARG);
  // CTAs per unit: about one per SM over the whole grid (a CTA's fixed cost is
  // several tiles' worth), at most one per cache tile of the longest sequence.
  const int sms = mars_host::num_sms();
  const int max_tiles = std::max(1, ceil_div(max_len, kTileKeys));
  int cl = pow2_ceil(std::max(1, ceil_div(sms, units)));
  cl = std::min(cl, kMaxCluster);
  while (cl > 1 && cl > max_tiles) cl >>= 1;
  // Small units (<= 32 rows, the four-quarter path) with few units in the grid take
  // 16 CTAs each when the tiles allow: half the tiles per CTA for the same merge
  // (batch 1 of the 7B shape: 10.3 -> 10.1 us at cache 2048, 11.5 -> 10.9 at 3068).
  // The launch falls back to 8 where the device cannot schedule 16-CTA clusters.
  if (cl == kMaxCluster && a.Gc * S <= 32 && max_tiles >= kWideCluster && units * kWideCluster <= 2 * sms)
    cl = kWideCluster;
  a.C = cl;
  a.sort_units = (batch > 1 && batch <= kSortLimit) ? 1 : 0;
  a.box_rows = std::min(cap, kTileKeys);

  Maps mp;
  const long long dq[4] = {D, Hq, S, batch}, dc[4] = {D, cap, Hkv, batch}, dn[4] = {D, Hkv, S, batch};
  if (!make_map(&mp.q, q, dq, a.Gc, S) || !make_map(&mp.kc, k_cache, dc, a.box_rows, 1) ||
      !make_map(&mp.vc, v_cache, dc, a.box_rows, 1) || !make_map(&mp.kn, k_new, dn, 1, S) ||
      !make_map(&mp.vn, v_new, dn, 1, S))
    return MARS_ERR_CUDA;
  const bool small = a.Gc * S <= 32 && a.C > 1;
  if (D == 64)
    return small ? launch<64, true>(mp, a, static_cast<int>(units), stream)
                 : launch<64, false>(mp, a, static_cast<int>(units), stream);
  return small ? launch<128, true>(mp, a, static_cast<int>(units), stream)
               : launch<128, false>(mp, a, static_cast<int>(units), stream);
}

}  // namespace

extern "C" size_t mars_decode_attn_workspace_size(int, int, int, int, int) { return 0; }

extern "C" int mars_decode_attn(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                                const uint16_t* k_cache, const uint16_t* v_cache, const int32_t* cache_len, int batch,
                                int B, int Hq, int Hkv, int D, int cap, int max_len, float scale, uint16_t* o,
                                int32_t* status, void* stream) {
  return decode_impl(q, k_new, v_new, k_cache, v_cache, nullptr, nullptr, cache_len, nullptr, batch, B, Hq, Hkv, D,
                     cap, max_len, scale, o, status, static_cast<cudaStream_t>(stream));
}

extern "C" int mars_decode_attn_deferred(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                                         uint16_t* k_cache, uint16_t* v_cache, const int32_t* cache_len,
                                         const int32_t* pending, int batch, int B, int Hq, int Hkv, int D, int cap,
                                         int max_len, float scale, uint16_t* o, int32_t* status, void* stream) {
  MARS_HOST_CHECK(pending != nullptr, MARS_ERR_INVALID_ARG);
  return decode_impl(q, k_new, v_new, k_cache, v_cache, k_cache, v_cache, cache_len, pending, batch, B, Hq, Hkv, D,
                     cap, max_len, scale, o, status, static_cast<cudaStream_t>(stream));
}
