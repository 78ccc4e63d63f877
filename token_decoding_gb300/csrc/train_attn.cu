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
// tiles inside every row's interval take no mask, and the rest take a
// two-compare interval mask.
//
// sm_103a design (one CTA per (batch, head, 128-row query tile)):
//   warp 0      TMA producer: Q once, then K and V tiles (SW128, 64-column
//               boxes) into an NS-stage ring with full/empty mbarriers.
//   warp 1      TMEM owner and MMA issuer (one thread): S = Q K^T into one of
//               two 128-column TMEM buffers, O += P V into a D-column TMEM
//               accumulator; completion is signalled with tcgen05.commit.
//   warps 2..5  softmax (thread = query row = TMEM lane): S from TMEM, mask,
//               row max, exp2, P (bf16) into shared memory in the K-major
//               SW128 layout the PV MMA reads (on partial tiles as a hi + lo
//               pair of bf16 terms, two PV passes); O in TMEM is rescaled only when
//               the row max grew by more than 2^8 (lazy rescaling), and the
//               epilogue normalises O and stores bf16 (and the log-sum-exp).
// The MMA warp issues S(n) before PV(n-1), so the tensor cores compute the
// next scores while the softmax warps work on the current ones.
// Every mbarrier wait is bounded; a wait that gives up sets MARS_DEV_TIMEOUT
// in the status word and the CTA winds down without further waiting.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace {

using namespace mars;

constexpr int kBM = 128;        // query rows per CTA
constexpr int kBN = 128;        // keys per tile
constexpr int kBox = 128 * 128; // bytes of one [128 rows x 64 bf16] SW128 box
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P values stay below 2^8

template <int D>
struct Cfg {
  static constexpr int NB = D / 64;  // 64-column boxes per row block
  static constexpr int NS = D == 64 ? 3 : 2;
  static constexpr int Q_BYTES = NB * kBox;
  static constexpr int KV_BYTES = NB * kBox;  // one K (or V) tile
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + Q_BYTES;
  static constexpr int V_OFF = K_OFF + NS * KV_BYTES;
  static constexpr int P_OFF = V_OFF + NS * KV_BYTES;
  static constexpr int P_BYTES = 2 * kBox;
  static constexpr int PLO_OFF = P_OFF + P_BYTES;       // low bf16 part of P on partial tiles
  static constexpr int SMEM = PLO_OFF + P_BYTES + 1024;  // + slack to align the base to 1024
  static constexpr int TMEM_COLS = 512;                 // S0 | S1 | O
  static constexpr int O_COL = 2 * kBN;
};

struct TrainArgs {
  uint16_t* o;
  float* lse;
  int32_t* status;
  int batch, L, B, Hq, Hkv, G;
  float scale_log2;
  int nq;         // query tiles per stream
};

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
  __device__ __forceinline__ int count() const { return n_clean + n_noisy; }
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

__device__ __forceinline__ Sched make_sched(bool noisy_q, int j, int L, int B) {
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

template <int D>
__global__ void __launch_bounds__(192, 1)
    train_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const TrainArgs a) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar_q, bar_k[C::NS], bar_v[C::NS], bar_kv_empty[C::NS], bar_s[2], bar_p,
      bar_pv;
  __shared__ uint32_t tmem_slot;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- which query tile: heaviest first (noisy j, clean j for j = nq-1 .. 0), heads innermost
  const int bh_count = a.batch * a.Hq;
  const int rank = blockIdx.x / bh_count;
  const int bh = blockIdx.x % bh_count;
  const int b = bh / a.Hq, h = bh % a.Hq, g = h / a.G;
  const int j = a.nq - 1 - rank / 2;
  const bool noisy_q = (rank & 1) == 0;
  const int r0 = noisy_q ? a.L + kBM * j : kBM * j;   // first z row of the tile
  const int row_end = noisy_q ? 2 * a.L : a.L;       // rows at or past this are not stored
  const Sched sched = make_sched(noisy_q, j, a.L, a.B);
  const int ntiles = sched.count();

  if (threadIdx.x == 0) {
    mbar_init(&bar_q, 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&bar_k[s], 1);
      mbar_init(&bar_v[s], 1);
      mbar_init(&bar_kv_empty[s], 1);
    }
    mbar_init(&bar_s[0], 1);
    mbar_init(&bar_s[1], 1);
    mbar_init(&bar_p, 128);
    mbar_init(&bar_pv, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  const uint32_t q_s = smem_u32(smem + C::Q_OFF);
  const uint32_t k_s = smem_u32(smem + C::K_OFF);
  const uint32_t v_s = smem_u32(smem + C::V_OFF);
  const uint32_t p_s = smem_u32(smem + C::P_OFF);
  const uint32_t plo_s = smem_u32(smem + C::PLO_OFF);

  if (warp == 0) {
    // ================= TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&bar_q, C::Q_BYTES);
      for (int c = 0; c < C::NB; ++c) tma_load_4d(q_s + c * kBox, &tm_q, &bar_q, 64 * c, h, r0, b);
      for (int n = 0; n < ntiles; ++n) {
        const int st = n % C::NS;
        if (n >= C::NS && !mbar_wait(&bar_kv_empty[st], ((n / C::NS) - 1) & 1)) {
          set_status(a.status, MARS_DEV_TIMEOUT);
          break;
        }
        int kstart;
        bool nz, part;
        sched.at(n, kstart, nz, part);
        mbar_arrive_expect_tx(&bar_k[st], C::KV_BYTES);
        for (int c = 0; c < C::NB; ++c)
          tma_load_4d(k_s + st * C::KV_BYTES + c * kBox, &tm_k, &bar_k[st], 64 * c, g, kstart, b);
        mbar_arrive_expect_tx(&bar_v[st], C::KV_BYTES);
        for (int c = 0; c < C::NB; ++c)
          tma_load_4d(v_s + st * C::KV_BYTES + c * kBox, &tm_v, &bar_v[st], 64 * c, g, kstart, b);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_bf16(kBM, kBN, false);
      constexpr uint32_t id_pv = idesc_bf16(kBM, D, true);
      bool ok = mbar_wait(&bar_q, 0);
      auto issue_pv = [&](int n) {
        const int st = n % C::NS;
        ok = ok && mbar_wait(&bar_p, n & 1);
        ok = ok && mbar_wait(&bar_v[st], (n / C::NS) & 1);
        if (!ok) return;
        int kstart;
        bool nz, part;
        sched.at(n, kstart, nz, part);
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks) {
          const uint64_t ad = smem_desc(p_s + (ks >> 2) * kBox + (ks & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc(v_s + st * C::KV_BYTES + ks * 16 * 128, kBox, 1024);
          tc_mma_ss(tmem + C::O_COL, ad, bd, id_pv, (n > 0 || ks > 0) ? 1u : 0u);
        }
        if (part) {  // second pass with the low bf16 part of P
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks) {
            const uint64_t ad = smem_desc(plo_s + (ks >> 2) * kBox + (ks & 3) * 32, 16, 1024);
            const uint64_t bd = smem_desc(v_s + st * C::KV_BYTES + ks * 16 * 128, kBox, 1024);
            tc_mma_ss(tmem + C::O_COL, ad, bd, id_pv, 1u);
          }
        }
        tc_commit(&bar_pv);
        tc_commit(&bar_kv_empty[st]);
      };
      for (int n = 0; ok && n < ntiles; ++n) {
        const int st = n % C::NS;
        ok = mbar_wait(&bar_k[st], (n / C::NS) & 1);
        if (!ok) break;
        tc_fence_after();
        const uint32_t s_col = (n & 1) * kBN;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t ad = smem_desc(q_s + (ks >> 2) * kBox + (ks & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc(k_s + st * C::KV_BYTES + (ks >> 2) * kBox + (ks & 3) * 32, 16, 1024);
          tc_mma_ss(tmem + s_col, ad, bd, id_qk, ks > 0 ? 1u : 0u);
        }
        tc_commit(&bar_s[n & 1]);
        if (n > 0) issue_pv(n - 1);
      }
      if (ok) issue_pv(ntiles - 1);
      if (!ok) set_status(a.status, MARS_DEV_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ================= softmax / epilogue (warps 2..5, thread = row)
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const int i = r0 + r;  // z position of this row
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    // visible key intervals of this row: clean [c_lo_v, c_hi_v], noisy [n_lo_v, n_hi_v]
    int c_hi_v, n_lo_v, n_hi_v;
    if (i < a.L) {
      c_hi_v = i;
      n_lo_v = 1;
      n_hi_v = 0;
    } else {
      const int t = i - a.L;
      const int c = a.B * (t / a.B);
      c_hi_v = c - 1;
      n_lo_v = a.L + c;
      n_hi_v = i;
    }
    float m_used = -INFINITY;  // max the current P values are relative to
    float l = 0.f;
    bool ok = true;
    uint8_t* p_row = smem + C::P_OFF + r * 128;
    uint8_t* plo_row = smem + C::PLO_OFF + r * 128;
    const int sw = r & 7;

    for (int n = 0; n < ntiles; ++n) {
      int kstart;
      bool nz, part;
      sched.at(n, kstart, nz, part);
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_s[n & 1], (n >> 1) & 1));
      if (!ok) break;
      tc_fence_after();
      uint32_t s[kBN];
#pragma unroll
      for (int c = 0; c < kBN; c += 16) {
        uint32_t (&chunk)[16] = *reinterpret_cast<uint32_t(*)[16]>(&s[c]);
        tmem_ld16(tmem + lane_addr + (n & 1) * kBN + c, chunk);
      }
      tc_wait_ld();
      // mask and row max on the raw scores (scale > 0 commutes with max)
      float mx0 = -INFINITY, mx1 = -INFINITY;
      if (part) {
        const int lo = nz ? n_lo_v : 0;
        const int hi = nz ? n_hi_v : c_hi_v;
#pragma unroll
        for (int c = 0; c < kBN; ++c) {
          const int key = kstart + c;
          const float x = (key >= lo && key <= hi) ? __uint_as_float(s[c]) : -INFINITY;
          s[c] = __float_as_uint(x);
          if (c & 1) mx1 = fmaxf(mx1, x);
          else mx0 = fmaxf(mx0, x);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kBN; c += 2) {
          mx0 = fmaxf(mx0, __uint_as_float(s[c]));
          mx1 = fmaxf(mx1, __uint_as_float(s[c + 1]));
        }
      }
      const float tile_max = fmaxf(mx0, mx1) * a.scale_log2;
      // lazy rescale: keep the old reference max unless the new one is 2^8 larger
      float alpha = 1.f;
      const bool grow = tile_max > m_used + kRescaleThreshold;
      if (grow) {
        alpha = fast_exp2(m_used - tile_max);  // 0 when m_used is -inf
        m_used = tile_max;
      }
      const float mu = m_used == -INFINITY ? 0.f : m_used;
      const float neg_mu = -mu;
      // P = exp2(s * scale_log2 - mu), kept in fp32 until the P buffer is free
      float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
      for (int c = 0; c < kBN; c += 2) {
        const float p0 = fast_exp2(fmaf(__uint_as_float(s[c]), a.scale_log2, neg_mu));
        const float p1 = fast_exp2(fmaf(__uint_as_float(s[c + 1]), a.scale_log2, neg_mu));
        sum0 += p0;
        sum1 += p1;
        s[c] = __float_as_uint(p0);
        s[c + 1] = __float_as_uint(p1);
      }
      l = l * alpha + (sum0 + sum1);
      // PV(n-1) must be done before O is rescaled and before P is overwritten
      if (n > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_pv, (n - 1) & 1));
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
          for (int c = 0; c < D; c += 16) {
            uint32_t ov[16];
            tmem_ld16(tmem + lane_addr + C::O_COL + c, ov);
            tc_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st16(tmem + lane_addr + C::O_COL + c, ov);
          }
          tc_wait_st();
        }
      }
      // P row -> shared memory, K-major SW128: keys 64*sub + 8*cc .. +7 at chunk cc ^ (r & 7).
      // On partial tiles P is also split as hi + lo (two bf16 terms): rows that see only a
      // few keys have no averaging to hide the 2^-9 relative rounding of a single bf16 P.
#pragma unroll
      for (int c = 0; c < kBN / 8; ++c) {
        const int sub = c >> 3, cc = c & 7;
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = __uint_as_float(s[8 * c + 2 * e]), p1 = __uint_as_float(s[8 * c + 2 * e + 1]);
          hi[e] = pack_bf16x2(p0, p1);
          lo[e] = pack_bf16x2(p0 - bf16lo_to_f32(hi[e]), p1 - bf16hi_to_f32(hi[e]));
        }
        const int off = sub * kBox + ((cc ^ sw) << 4);
        *reinterpret_cast<uint4*>(p_row + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        if (part) *reinterpret_cast<uint4*>(plo_row + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&bar_p);
    }

    // ---- epilogue: O / l -> bf16, log-sum-exp
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bar_pv, (ntiles - 1) & 1));
    if (ok) {
      tc_fence_after();
      const float inv = 1.f / l;
      const bool store = i < row_end;
      uint16_t* dst = a.o + ((static_cast<size_t>(b) * 2 * a.L + i) * a.Hq + h) * D;
#pragma unroll
      for (int c = 0; c < D; c += 16) {
        uint32_t ov[16];
        tmem_ld16(tmem + lane_addr + C::O_COL + c, ov);
        tc_wait_ld();
        if (store) {
          uint4 w0 = make_uint4(pack_bf16x2(__uint_as_float(ov[0]) * inv, __uint_as_float(ov[1]) * inv),
                                pack_bf16x2(__uint_as_float(ov[2]) * inv, __uint_as_float(ov[3]) * inv),
                                pack_bf16x2(__uint_as_float(ov[4]) * inv, __uint_as_float(ov[5]) * inv),
                                pack_bf16x2(__uint_as_float(ov[6]) * inv, __uint_as_float(ov[7]) * inv));
          uint4 w1 = make_uint4(pack_bf16x2(__uint_as_float(ov[8]) * inv, __uint_as_float(ov[9]) * inv),
                                pack_bf16x2(__uint_as_float(ov[10]) * inv, __uint_as_float(ov[11]) * inv),
                                pack_bf16x2(__uint_as_float(ov[12]) * inv, __uint_as_float(ov[13]) * inv),
                                pack_bf16x2(__uint_as_float(ov[14]) * inv, __uint_as_float(ov[15]) * inv));
          *reinterpret_cast<uint4*>(dst + c) = w0;
          *reinterpret_cast<uint4*>(dst + c + 8) = w1;
        }
      }
      if (store && a.lse != nullptr)
        a.lse[(static_cast<size_t>(b) * a.Hq + h) * 2 * a.L + i] = (m_used + __log2f(l)) * 0.6931471805599453f;
    } else if (lane == 0) {
      set_status(a.status, MARS_DEV_TIMEOUT);
    }
    tc_fence_before();
  }

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

// [batch, n, H, D] bf16 viewed as a 4-D tensor with 64-column x 128-row SW128 boxes.
bool make_map(CUtensorMap* m, const void* ptr, int D, int H, int n, int batch) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(n),
                              static_cast<cuuint64_t>(batch)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2,
                                 static_cast<cuuint64_t>(n) * H * D * 2};
  const cuuint32_t box[4] = {64, 1, 128, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
int launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const TrainArgs& a,
           cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(train_attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::SMEM) !=
        cudaSuccess)
      return MARS_ERR_CUDA;
    configured = true;
  }
  const long long grid = static_cast<long long>(a.batch) * a.Hq * 2 * a.nq;
  train_attn_kernel<D><<<static_cast<unsigned>(grid), 192, Cfg<D>::SMEM, stream>>>(tq, tk, tv, a);
  return cudaGetLastError() == cudaSuccess ? MARS_OK : MARS_ERR_CUDA;
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

  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, q, D, Hq, 2 * L, batch) || !make_map(&tk, k, D, Hkv, 2 * L, batch) ||
      !make_map(&tv, v, D, Hkv, 2 * L, batch))
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
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return D == 64 ? launch<64>(tq, tk, tv, a, s) : launch<128>(tq, tk, tv, a, s);
}
