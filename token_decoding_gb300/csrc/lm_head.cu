// lm_head.cu - the LM head of the proposal positions fused with the row
// reduction of the acceptance step: logits = hidden . weight^T are computed
// tile by tile in tensor memory and reduced on the spot to each row's
// (max, lowest argmax, sum of exp); the logits never reach global memory.
//
// Method: the authors' MARS blog post, "Where it stands against the
// alternatives" (every proposal ends in the 152k-vocabulary projection, the
// drafter's cost) and "Inference: a knob, not a mode switch" (the top-1
// probability gate that reads those logits).
//
// sm_103a design (tensor-bound for a full batch of proposals, HBM-bound for a
// handful): a CTA takes one 128-row tile of hidden states and a contiguous
// range of 256-row tiles of the weight (vocabulary entries).  For each weight
// tile the K loop runs tcgen05.mma M128 N256 K16 over 64-column SW128 boxes of
// both operands (TMA, NS-stage ring) into one of two tensor-memory
// accumulators, so the reduction of tile j overlaps the products of tile j + 1.
//   warp 0      TMA producer (hidden box [128 x 64], weight box [256 x 64]);
//   warp 1      tensor-memory owner and MMA issuer (one elected lane);
//   warps 2..9  reduction: thread = row (lane quarter of its warp), warps 2..5
//               take columns 0..127 of a tile, warps 6..9 columns 128..255;
//               each keeps a running (max, lowest index of the max, sum of
//               exp(x - max)) over its columns of every tile of the range.
// The CTA writes one partial per (row, vocabulary range), in the layout of the
// acceptance step's partials, so the acceptance's finish merges them.  The CTAs
// that share a vocabulary range are adjacent in launch order and read the
// same weight tiles at about the same time (one HBM read, the rest from L2).
// Every mbarrier wait is bounded; a wait that gives up sets MARS_DEV_TIMEOUT.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "lm_head.cuh"

namespace {

using namespace mars;

constexpr int kBM = 128;            // hidden rows per tile
constexpr int kBN = 256;            // vocabulary entries per weight tile
constexpr int kBK = 64;             // K per stage (one SW128 box column)
constexpr int kNS = 4;              // ring stages
constexpr int kABox = kBM * 128;    // bytes of one hidden box [128 x 64]
constexpr int kBBox = kBN * 128;    // bytes of one weight box [256 x 64]
constexpr int kStage = kABox + kBBox;
constexpr int kSmem = kNS * kStage + 1024;  // + slack to align the base to 1024
constexpr int kThreads = 320;
constexpr int kTmemCols = 2 * kBN;  // two accumulators

struct HeadArgs {
  float4* partials;  // [M][nsplit]: (max, argmax bits, sum of exp(x - max), -inf)
  int32_t* status;
  int M, K, V;
  int mtiles, nsplit, ntiles;  // hidden tiles, vocabulary ranges, weight tiles
};

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;  // descriptor version for sm_100-class tensor cores
  d |= 2ull << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor: bf16 x bf16 -> fp32, dense, M x N, A and B K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// (m, idx, s) <- merge with (m2, i2, s2): larger max wins, equal maxima keep the lower index.
__device__ __forceinline__ void merge_state(float& m, int& idx, float& s, float m2, int i2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    idx = i2;
    s = s2;
  } else if (m2 > m) {
    s = s * fast_exp2((m - m2) * kLog2e) + s2;
    m = m2;
    idx = i2;
  } else if (m2 < m) {
    s += s2 * fast_exp2((m2 - m) * kLog2e);
  } else {
    s += s2;
    idx = min(idx, i2);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    lm_head_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w,
                   const HeadArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[kNS], empty[kNS], acc_full[2], acc_empty[2];
  __shared__ uint32_t tmem_slot;
  __shared__ float s_m[kBM], s_s[kBM];
  __shared__ int s_i[kBM];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = blockIdx.x % a.mtiles, sp = blockIdx.x / a.mtiles;
  const int j0 = static_cast<int>((static_cast<long long>(a.ntiles) * sp) / a.nsplit);
  const int j1 = static_cast<int>((static_cast<long long>(a.ntiles) * (sp + 1)) / a.nsplit);
  const int nk = a.K / kBK;
  if (tid == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&acc_full[x], 1);
      mbar_init(&acc_empty[x], 256);
    }
    fence_mbar_init();
    tma_prefetch_desc(&tm_h);
    tma_prefetch_desc(&tm_w);
  }
  if (warp == 1) tmem_alloc(&tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  // launched as a programmatic dependent: nothing global is read before the previous
  // kernel in the stream has completed; the acceptance finish that follows may start
  // once this wait has passed (it reads only what the kernel before this one wrote)
  griddep_wait();
  griddep_launch_dependents();
  const uint32_t ring = smem_u32(smem);
  bool ok = true;

  if (warp == 0) {
    // ================= TMA producer
    if (lane == 0) {
      int it = 0;
      for (int j = j0; j < j1 && ok; ++j)
        for (int kc = 0; kc < nk; ++kc, ++it) {
          const int st = it % kNS;
          if (it >= kNS && !mbar_wait(&empty[st], ((it / kNS) - 1) & 1)) {
            ok = false;
            break;
          }
          const uint32_t ab = ring + st * kStage, bb = ab + kABox;
          mbar_arrive_expect_tx(&full[st], kStage);
          tma_load_2d(ab, &tm_h, &full[st], kc * kBK, mt * kBM);
          tma_load_2d(bb, &tm_w, &full[st], kc * kBK, j * kBN);
        }
      if (!ok) set_status(a.status, MARS_DEV_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer: the whole warp runs the schedule (warp-uniform
    // descriptors); one elected lane issues the products and their commits
    const bool leader = elect_one();
    constexpr uint32_t idesc = idesc_bf16(kBM, kBN);
    const uint64_t da = smem_desc(ring, 16, 1024), db = smem_desc(ring + kABox, 16, 1024);
    int it = 0;
    for (int j = j0; j < j1 && ok; ++j) {
      const int t = j - j0, ab = t & 1;
      if (t >= 2) ok = __all_sync(0xffffffffu, mbar_wait(&acc_empty[ab], ((t >> 1) - 1) & 1));
      if (!ok) break;
      tc_fence_after();
      for (int kc = 0; kc < nk; ++kc, ++it) {
        const int st = it % kNS;
        ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (it / kNS) & 1));
        if (!ok) break;
        tc_fence_after();
        if (leader) {
          const uint64_t so = static_cast<uint64_t>((st * kStage) >> 4);
#pragma unroll
          for (int ks = 0; ks < kBK / 16; ++ks)
            tc_mma_ss(tmem + ab * kBN, da + so + ((ks * 32) >> 4), db + so + ((ks * 32) >> 4), idesc,
                      (kc > 0 || ks > 0) ? 1u : 0u);
          tc_commit(&empty[st]);
          if (kc == nk - 1) tc_commit(&acc_full[ab]);
        }
        __syncwarp();
      }
    }
    if (!ok && leader) set_status(a.status, MARS_DEV_TIMEOUT);
    __syncwarp();
  } else {
    // ================= reduction of the accumulators
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;  // columns [128 half, 128 half + 128) of each tile
    const int r = quad * 32 + lane;    // row of the hidden tile (TMEM lane)
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    float m = -INFINITY, s = 0.f;
    int idx = 0x7fffffff;
    for (int j = j0; j < j1; ++j) {
      const int t = j - j0, ab = t & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&acc_full[ab], (t >> 1) & 1));
      if (!ok) break;
      tc_fence_after();
      uint32_t v[128];
#pragma unroll
      for (int c = 0; c < 128; c += 32)
        tmem_ld32(tmem + lane_addr + ab * kBN + half * 128 + c, *reinterpret_cast<uint32_t(*)[32]>(&v[c]));
      tc_wait_ld();
      tc_fence_before();
      mbar_arrive(&acc_empty[ab]);  // the accumulator may take the next tile's products
      // vocabulary entries past V are the zero rows of the weight box: they do not count
      const int v0 = j * kBN + half * 128;
      const int nvalid = min(128, a.V - v0);
      if (nvalid < 128) {
#pragma unroll
        for (int c = 0; c < 128; ++c) v[c] = c < nvalid ? v[c] : 0xFF800000u;  // -inf
      }
      float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; c += 8) {
        m0 = fmax3(m0, __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
        m1 = fmax3(m1, __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
        m2 = fmax3(m2, __uint_as_float(v[c + 4]), __uint_as_float(v[c + 5]));
        m3 = fmax3(m3, __uint_as_float(v[c + 6]), __uint_as_float(v[c + 7]));
      }
      const float tmax = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
      if (tmax == -INFINITY) continue;  // nothing valid in this tile's columns (and none before)
      if (tmax > m) {  // a new maximum: its lowest column in this tile, rescale the sum
        int found = 0;
#pragma unroll
        for (int c = 127; c >= 0; --c) found = __uint_as_float(v[c]) == tmax ? c : found;
        s = m == -INFINITY ? 0.f : s * fast_exp2((m - tmax) * kLog2e);
        m = tmax;
        idx = v0 + found;
      }
      const float mneg = -m * kLog2e;
      uint64_t acc2 = 0;
#pragma unroll
      for (int c = 0; c < 128; c += 2) {
        float x0, x1;
        fma2(__uint_as_float(v[c]), __uint_as_float(v[c + 1]), kLog2e, mneg, x0, x1);
        add2(acc2, fast_exp2(x0), fast_exp2(x1));
      }
      s += sum2(acc2);
    }
    // the two column halves of a row meet in shared memory; half 0 writes the partial
    if (half == 1) {
      s_m[r] = ok ? m : -INFINITY;
      s_s[r] = ok ? s : 0.f;
      s_i[r] = idx;
    }
    named_bar_sync(1, 256);
    if (half == 0) {
      if (ok) merge_state(m, idx, s, s_m[r], s_i[r], s_s[r]);
      const int row = mt * kBM + r;
      if (row < a.M)
        a.partials[static_cast<size_t>(row) * a.nsplit + sp] =
            make_float4(ok ? m : -INFINITY, __int_as_float(idx), ok ? s : 0.f, -INFINITY);
    }
    if (!ok && lane == 0) set_status(a.status, MARS_DEV_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
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

// A row-major [rows, K] bf16 matrix as a 2-D tensor, loaded in SW128 boxes of 64 x box_rows.
bool make_map(CUtensorMap* m, const void* ptr, int K, int rows, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace mars_lm_head {

int splits_for(int M, int V) {
  const int mtiles = (M + kBM - 1) / kBM;
  const int ntiles = (V + kBN - 1) / kBN;
  // about one CTA per SM of a GB300 (152): the ranges of a vocabulary split go to
  // adjacent CTAs, so the grid is mtiles x nsplit
  return std::max(1, std::min(ntiles, 152 / std::max(1, std::min(mtiles, 152))));
}

int launch_partials(const uint16_t* hidden, const uint16_t* weight, int M, int K, int V, float4* partials,
                    int nsplit, int32_t* status, cudaStream_t stream) {
  HeadArgs a;
  a.partials = partials;
  a.status = status;
  a.M = M;
  a.K = K;
  a.V = V;
  a.mtiles = (M + kBM - 1) / kBM;
  a.ntiles = (V + kBN - 1) / kBN;
  a.nsplit = nsplit;
  CUtensorMap th, tw;
  if (!make_map(&th, hidden, K, M, kBM) || !make_map(&tw, weight, K, V, kBN)) return MARS_ERR_CUDA;
  static int done[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MARS_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
      const cudaError_t e = cudaFuncSetAttribute(lm_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
      if (e != cudaSuccess) return mars_host::cuda_fail(e);
      done[dev] = 1;
    }
  }
  cudaLaunchConfig_t cfg = mars_host::pdl_config(dim3(a.mtiles * a.nsplit, 1, 1), dim3(kThreads, 1, 1), kSmem, stream);
  cudaLaunchAttribute attr[1];
  mars_host::pdl_attr(cfg, attr);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, lm_head_kernel, th, tw, a);
  return e == cudaSuccess ? MARS_OK : mars_host::cuda_fail(e);
}

}  // namespace mars_lm_head
