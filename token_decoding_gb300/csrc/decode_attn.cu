// decode_attn.cu - mars_decode_attn: the B appended [MASK] queries of one
// sliding-window decode step attend to their sequence's committed KV cache
// and causally to each other.
//
// Method: "MARS: Enabling Autoregressive Models Multi-Token Generation",
// Fig. 2 (right, sliding-window inference: B placeholders appended after the
// cursor, filled by one forward) and Eq. 2 (noisy intra-block causal case);
// the authors' MARS blog post, "Inference: a knob, not a mode switch".
//
// Design (HBM-bound: every cached K/V byte is read once):
//   * A work unit is (sequence b, KV head g, chunk of Gc query heads of that
//     group).  Its query rows are (head, position) pairs, R = Gc * B <= 128,
//     so one K/V stream serves all heads that share the KV head (GQA).
//   * A unit is processed by a cluster of C CTAs; CTA rank r takes the r-th
//     contiguous share of the unit's 64-key tiles (committed keys followed by
//     this step's B new keys).  Each CTA keeps an online softmax state per
//     row; at the end the C states are merged through distributed shared
//     memory, so no split-K workspace ever reaches global memory.
//   * K/V tiles are streamed with cp.async (16-byte, XOR-swizzled rows) in a
//     3-stage ring; Q K^T and P V run on bf16 mma.sync with fp32 accumulation,
//     softmax in the exp2 domain with fp32 state.
//   * Units are visited longest-cache-first (a rank computed in every CTA from
//     cache_len), so the long sequences start early and short ones fill in.
#include <algorithm>

#include "common.cuh"

namespace {

using namespace mars;

constexpr int kTileKeys = 64;
constexpr int kStages = 3;
constexpr int kMaxRows = 128;
constexpr int kMaxCluster = 8;
constexpr int kSortLimit = 256;  // sequences; above this units are visited in index order

struct DecodeArgs {
  const uint16_t* q;
  const uint16_t* k_new;
  const uint16_t* v_new;
  const uint16_t* k_cache;
  const uint16_t* v_cache;
  const int32_t* cache_len;
  uint16_t* o;
  int32_t* status;
  int batch, B, Hq, Hkv, cap, max_len;
  float scale_log2;  // scale * log2(e)
  int G;             // Hq / Hkv
  int Gc;            // query heads per unit
  int nhc;           // head chunks per KV head
  int C;             // CTAs per unit (cluster size)
  int sort_units;
};

template <int D>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  // byte offset of 16-byte chunk `chunk` of row `row` in a [rows x D] bf16 tile
  return static_cast<uint32_t>(row * (D * 2) + ((chunk ^ (row & 7)) << 4));
}

template <int D, int NW>
__global__ void __launch_bounds__(NW * 32) decode_kernel(const DecodeArgs a) {
  constexpr int RP = NW * 16;           // padded rows
  constexpr int NT = NW * 32;           // threads
  constexpr int CPR = D / 8;            // 16-byte chunks per row
  constexpr int KT = D / 16;            // k-steps of Q K^T
  constexpr int DT = D / 8;             // n-tiles of P V
  constexpr uint32_t kTileBytes = kTileKeys * D * 2;

  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* q_s = smem;
  uint8_t* kv_s = smem + RP * D * 2;  // [stage][K tile | V tile]
  __shared__ int s_b;
  __shared__ int s_len[kSortLimit];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int units_per_b = a.Hkv * a.nhc;
  const int unit_rank = blockIdx.x / a.C;
  const int crank = a.C > 1 ? static_cast<int>(cluster_ctarank()) : 0;

  // ---- which sequence: heavy-first rank order (stable by index) or plain order
  const int b_rank = unit_rank / units_per_b;
  if (a.sort_units) {
    for (int t = tid; t < a.batch; t += NT) s_len[t] = __ldg(a.cache_len + t);
    __syncthreads();
    for (int t = tid; t < a.batch; t += NT) {
      const int lt = s_len[t];
      int rank = 0;
      for (int u = 0; u < a.batch; ++u) {
        const int lu = s_len[u];
        rank += (lu > lt) || (lu == lt && u < t);
      }
      if (rank == b_rank) s_b = t;
    }
    __syncthreads();
  } else {
    if (tid == 0) s_b = b_rank;
    __syncthreads();
  }
  const int b = s_b;
  const int rem = unit_rank % units_per_b;
  const int g = rem / a.nhc;
  const int hc = rem % a.nhc;
  const int h0 = g * a.G + hc * a.Gc;                // first query head of this unit
  const int heads = min(a.Gc, a.G - hc * a.Gc);      // heads in this unit
  const int R = heads * a.B;                         // real rows

  const int len = __ldg(a.cache_len + b);
  if (len < 0 || len > a.max_len) {
    // Uniform over the cluster: every CTA of the unit sees the same len and returns here.
    if (crank == 0) {
      if (tid == 0) set_status(a.status, MARS_DEV_LEN_RANGE);
      for (int e = tid; e < R * CPR; e += NT) {
        const int r = e / CPR, c = e % CPR;
        const int hl = r / a.B, i = r % a.B;
        *reinterpret_cast<uint4*>(a.o + ((static_cast<size_t>(b) * a.B + i) * a.Hq + h0 + hl) * D + 8 * c) =
            make_uint4(0, 0, 0, 0);
      }
    }
    return;
  }
  const int T = len + a.B;  // keys: committed cache + this step's placeholders
  const int ntiles = (T + kTileKeys - 1) / kTileKeys;
  const int t0 = static_cast<int>((static_cast<long long>(ntiles) * crank) / a.C);
  const int t1 = static_cast<int>((static_cast<long long>(ntiles) * (crank + 1)) / a.C);

  const size_t cache_head = (static_cast<size_t>(b) * a.Hkv + g) * a.cap;  // row index of (b, g, 0)

  // ---- Q tile -> smem (rows beyond R are zero)
  const uint32_t q_base = smem_u32(q_s);
  for (int e = tid; e < RP * CPR; e += NT) {
    const int r = e / CPR, c = e % CPR;
    const bool valid = r < R;
    const int hl = valid ? r / a.B : 0, i = valid ? r % a.B : 0;
    const uint16_t* src = a.q + ((static_cast<size_t>(b) * a.B + i) * a.Hq + h0 + hl) * D + 8 * c;
    cp_async16(q_base + swz<D>(r, c), src, valid);
  }
  cp_async_commit();

  const uint32_t kv_base = smem_u32(kv_s);
  auto load_tile = [&](int tile, int stage) {
    const uint32_t kb = kv_base + stage * 2 * kTileBytes;
    const uint32_t vb = kb + kTileBytes;
    for (int e = tid; e < kTileKeys * CPR; e += NT) {
      const int r = e / CPR, c = e % CPR;
      const int key = tile * kTileKeys + r;
      const uint16_t* ks;
      const uint16_t* vs;
      bool valid = true;
      if (key < len) {
        ks = a.k_cache + (cache_head + key) * D + 8 * c;
        vs = a.v_cache + (cache_head + key) * D + 8 * c;
      } else if (key < T) {
        const size_t off = ((static_cast<size_t>(b) * a.B + (key - len)) * a.Hkv + g) * D + 8 * c;
        ks = a.k_new + off;
        vs = a.v_new + off;
      } else {
        ks = a.k_new;
        vs = a.v_new;
        valid = false;
      }
      cp_async16(kb + swz<D>(r, c), ks, valid);
      cp_async16(vb + swz<D>(r, c), vs, valid);
    }
  };

#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (t0 + s < t1) load_tile(t0 + s, s);
    cp_async_commit();
  }

  // ---- per-warp state: rows warp*16 + lane/4 (+8)
  float m_r[2] = {-INFINITY, -INFINITY};
  float l_r[2] = {0.f, 0.f};
  float acc[DT][4];
#pragma unroll
  for (int n = 0; n < DT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
  uint32_t qf[KT][4];
  const int row0 = warp * 16 + (lane >> 2);
  const int i_row[2] = {row0 % a.B, (row0 + 8) % a.B};

  cp_async_wait<kStages - 2>();
  __syncthreads();
#pragma unroll
  for (int kk = 0; kk < KT; ++kk) {
    const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int c = 2 * kk + (lane >> 4);
    ldsm_x4(q_base + swz<D>(r, c), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
  }

  for (int tile = t0; tile < t1; ++tile) {
    const int it = tile - t0;
    cp_async_wait<kStages - 2>();
    __syncthreads();
    {
      const int nt = tile + kStages - 1;
      if (nt < t1) load_tile(nt, (it + kStages - 1) % kStages);
      cp_async_commit();
    }
    const uint32_t kb = kv_base + (it % kStages) * 2 * kTileBytes;
    const uint32_t vb = kb + kTileBytes;

    // S = Q K^T  (16 rows x 64 keys per warp)
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
#pragma unroll
      for (int j2 = 0; j2 < 4; ++j2) {
        uint32_t b0, b1, b2, b3;
        const int r = 16 * j2 + (lane & 7) + (lane >> 4) * 8;
        const int c = 2 * kk + ((lane >> 3) & 1);
        ldsm_x4(kb + swz<D>(r, c), b0, b1, b2, b3);
        mma_bf16_16816(s[2 * j2], qf[kk], b0, b1);
        mma_bf16_16816(s[2 * j2 + 1], qf[kk], b2, b3);
      }
    }

    // mask (keys past len + i are invisible) and online softmax in the exp2 domain
    const int kbase = tile * kTileKeys + 2 * (lane & 3);
    const bool need_mask = tile * kTileKeys + kTileKeys - 1 > len;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hr = e >> 1;
        float x = s[j][e] * a.scale_log2;
        if (need_mask && kbase + 8 * j + (e & 1) > len + i_row[hr]) x = -INFINITY;
        s[j][e] = x;
        mx[hr] = fmaxf(mx[hr], x);
      }
    }
    float alpha[2], mu[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 1));
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 2));
      const float mnew = fmaxf(m_r[hr], mx[hr]);
      mu[hr] = mnew == -INFINITY ? 0.f : mnew;
      alpha[hr] = fast_exp2(m_r[hr] - mu[hr]);  // exp2(-inf) = 0 on the first visible tile
      m_r[hr] = mnew;
      l_r[hr] *= alpha[hr];
    }
#pragma unroll
    for (int n = 0; n < DT; ++n) {
      acc[n][0] *= alpha[0];
      acc[n][1] *= alpha[0];
      acc[n][2] *= alpha[1];
      acc[n][3] *= alpha[1];
    }
    uint32_t pf[4][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float p0 = fast_exp2(s[j][0] - mu[0]);
      const float p1 = fast_exp2(s[j][1] - mu[0]);
      const float p2 = fast_exp2(s[j][2] - mu[1]);
      const float p3 = fast_exp2(s[j][3] - mu[1]);
      l_r[0] += p0 + p1;
      l_r[1] += p2 + p3;
      // accumulator layout of n-tile j -> A-fragment layout of k-step j/2
      pf[j >> 1][(j & 1) * 2 + 0] = pack_bf16x2(p0, p1);
      pf[j >> 1][(j & 1) * 2 + 1] = pack_bf16x2(p2, p3);
    }

    // O += P V
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int dn = 0; dn < DT / 2; ++dn) {
        uint32_t b0, b1, b2, b3;
        const int r = 16 * kk + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = 2 * dn + (lane >> 4);
        ldsm_x4_t(vb + swz<D>(r, c), b0, b1, b2, b3);
        mma_bf16_16816(acc[2 * dn], pf[kk], b0, b1);
        mma_bf16_16816(acc[2 * dn + 1], pf[kk], b2, b3);
      }
    }
  }
  cp_async_wait<0>();

#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    l_r[hr] += __shfl_xor_sync(0xffffffffu, l_r[hr], 1);
    l_r[hr] += __shfl_xor_sync(0xffffffffu, l_r[hr], 2);
  }

  const int col0 = 2 * (lane & 3);
  if (a.C == 1) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = row0 + 8 * hr;
      if (r >= R) continue;
      const float inv = 1.f / l_r[hr];
      const int hl = r / a.B, i = r % a.B;
      uint16_t* dst = a.o + ((static_cast<size_t>(b) * a.B + i) * a.Hq + h0 + hl) * D;
#pragma unroll
      for (int n = 0; n < DT; ++n)
        *reinterpret_cast<uint32_t*>(dst + 8 * n + col0) = pack_bf16x2(acc[n][2 * hr] * inv, acc[n][2 * hr + 1] * inv);
    }
    return;
  }

  // ---- cluster merge through distributed shared memory
  __syncthreads();  // every warp is done with the K/V ring, which now holds the states
  float* acc_s = reinterpret_cast<float*>(kv_s);  // [RP][D]
  float* m_s = acc_s + RP * D;                     // [RP]
  float* l_s = m_s + RP;                           // [RP]
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int r = row0 + 8 * hr;
#pragma unroll
    for (int n = 0; n < DT; ++n) {
      acc_s[r * D + 8 * n + col0] = acc[n][2 * hr];
      acc_s[r * D + 8 * n + col0 + 1] = acc[n][2 * hr + 1];
    }
    if ((lane & 3) == 0) {
      m_s[r] = m_r[hr];
      l_s[r] = l_r[hr];
    }
  }
  cluster_sync();
  const uint32_t acc_local = smem_u32(acc_s), m_local = smem_u32(m_s), l_local = smem_u32(l_s);
  const int rows_per = (R + a.C - 1) / a.C;
  const int r_lo = crank * rows_per, r_hi = min(R, r_lo + rows_per);
  for (int e = tid; e < (r_hi - r_lo) * (D / 4); e += NT) {
    const int r = r_lo + e / (D / 4);
    const int d4 = e % (D / 4);
    float mmax = -INFINITY;
    for (int c = 0; c < a.C; ++c) mmax = fmaxf(mmax, dsmem_ld_f32(dsmem_map(m_local + 4 * r, c)));
    float l = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = 0; c < a.C; ++c) {
      const float mc = dsmem_ld_f32(dsmem_map(m_local + 4 * r, c));
      const float w = mc == -INFINITY ? 0.f : fast_exp2(mc - mmax);
      l += w * dsmem_ld_f32(dsmem_map(l_local + 4 * r, c));
      const float4 x = dsmem_ld_f32x4(dsmem_map(acc_local + 4 * (r * D + 4 * d4), c));
      o.x += w * x.x;
      o.y += w * x.y;
      o.z += w * x.z;
      o.w += w * x.w;
    }
    const float inv = 1.f / l;
    const int hl = r / a.B, i = r % a.B;
    uint16_t* dst = a.o + ((static_cast<size_t>(b) * a.B + i) * a.Hq + h0 + hl) * D + 4 * d4;
    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(o.x * inv, o.y * inv), pack_bf16x2(o.z * inv, o.w * inv));
  }
  cluster_sync();  // keep this CTA's shared memory alive until every peer has read it
}

template <int D, int NW>
size_t smem_bytes() {
  const size_t ring = static_cast<size_t>(kStages) * 2 * kTileKeys * D * 2;
  const size_t merge = static_cast<size_t>(NW * 16) * D * 4 + 2 * NW * 16 * 4;
  return static_cast<size_t>(NW * 16) * D * 2 + std::max(ring, merge);
}

template <int D, int NW>
int launch(const DecodeArgs& a, int units, cudaStream_t stream) {
  auto kern = decode_kernel<D, NW>;
  const size_t smem = smem_bytes<D, NW>();
  static bool configured = false;  // per instantiation; the attribute is process-wide
  if (!configured) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return mars_host::cuda_fail(e);
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(units * a.C, 1, 1);
  cfg.blockDim = dim3(NW * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return mars_host::cuda_fail(e);
  return MARS_OK;
}

template <int D>
int dispatch_rows(const DecodeArgs& a, int units, int rows, cudaStream_t s) {
  if (rows <= 16) return launch<D, 1>(a, units, s);
  if (rows <= 32) return launch<D, 2>(a, units, s);
  if (rows <= 64) return launch<D, 4>(a, units, s);
  return launch<D, 8>(a, units, s);
}

inline int ceil_div(long long x, long long y) { return static_cast<int>((x + y - 1) / y); }
inline int pow2_ceil(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

}  // namespace

extern "C" int mars_decode_attn(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                                const uint16_t* k_cache, const uint16_t* v_cache, const int32_t* cache_len, int batch,
                                int B, int Hq, int Hkv, int D, int cap, int max_len, float scale, uint16_t* o,
                                int32_t* status, void* stream) {
  using mars_host::aligned16;
  MARS_HOST_CHECK(batch > 0 && B >= 1 && B <= 16 && Hq > 0 && Hkv > 0 && Hq % Hkv == 0, MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(D == 64 || D == 128, MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(cap > 0 && max_len >= 0 && max_len <= cap, MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(scale > 0.f && scale < INFINITY, MARS_ERR_INVALID_ARG);
  const void* ptrs[] = {q, k_new, v_new, k_cache, v_cache, o};
  for (const void* p : ptrs) MARS_HOST_CHECK(p != nullptr && aligned16(p), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(cache_len != nullptr && mars_host::aligned4(cache_len), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(status == nullptr || mars_host::aligned4(status), MARS_ERR_INVALID_ARG);
  int rc = mars_host::check_device();
  if (rc != MARS_OK) return rc;

  DecodeArgs a;
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.cache_len = cache_len;
  a.o = o;
  a.status = status;
  a.batch = batch;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.cap = cap;
  a.max_len = max_len;
  a.scale_log2 = scale * kLog2e;
  a.G = Hq / Hkv;

  // Heads per unit: as many as fit in 128 rows, fewer when that leaves the GPU idle.
  const int sms = mars_host::num_sms();
  int Gc = std::min(a.G, kMaxRows / B);
  int nhc = ceil_div(a.G, Gc);
  const long long base_units = static_cast<long long>(batch) * Hkv;
  while (Gc > 1 && base_units * nhc * kMaxCluster < sms) {
    Gc = ceil_div(Gc, 2);
    nhc = ceil_div(a.G, Gc);
  }
  const long long units = base_units * nhc;
  MARS_HOST_CHECK(units * kMaxCluster < (1LL << 31), MARS_ERR_INVALID_ARG);
  const int max_tiles = ceil_div(static_cast<long long>(max_len) + B, kTileKeys);
  int C = pow2_ceil(std::max(1, ceil_div(2LL * sms, units)));
  C = std::min(C, kMaxCluster);
  while (C > 1 && C > max_tiles) C >>= 1;
  a.Gc = Gc;
  a.nhc = nhc;
  a.C = C;
  a.sort_units = (batch > 1 && batch <= kSortLimit) ? 1 : 0;

  const int rows = Gc * B;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return D == 64 ? dispatch_rows<64>(a, static_cast<int>(units), rows, s)
                 : dispatch_rows<128>(a, static_cast<int>(units), rows, s);
}
