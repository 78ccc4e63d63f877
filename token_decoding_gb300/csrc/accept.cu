// accept.cu - mars_accept: top-1 probability, greedy token, left-to-right
// commit with threshold tau, and the block-level KV append, in one call (a
// streaming launch and a finish launch).
//
// Method: the authors' MARS blog post, "Inference: a knob, not a mode switch"
// (commit while the top-1 probability holds, stop at the first position below
// tau); "MARS: Enabling Autoregressive Models Multi-Token Generation",
// Sec. 3.1 gap (4) (strictly left to right) and its block-level KV cache
// contribution; the aitrends.kr summary (at least one token is accepted).
//
// Design (HBM-bound: one read of the logits, no atomics, no counters):
//   * Launch 1 (accept_kernel).  Each row (b, i) of logits is cut into 16 KB
//     chunks; a chunk is one work item.  CTAs are persistent, one per SM: CTA c
//     takes items c, c + grid, ...  A producer warp streams the CTA's chunks
//     with 1-D bulk copies (cp.async.bulk) into a ring of kSlots 16 KB
//     shared-memory slots guarded by full/empty mbarriers (~190 KB in flight
//     per SM).  Consumer warp w owns slot w and takes every kSlots-th chunk:
//     its lanes read 16-byte vectors from the slot, take the group max on
//     packed bf16, keep the group that raised the running max in registers
//     (one argmax scan per lane and chunk), and accumulate
//     sum exp2(x*log2e - max*log2e) with packed fp32x2 FMA/ADD.  The slot is
//     released as soon as it is read; the warp reduces with shuffles and
//     stores the chunk's (max, argmax, sum) partial.
//   * Launch 2 (accept_finish_kernel, programmatic dependent launch: it starts
//     while launch 1 runs, prefetches cache_len and the candidate K/V rows, and
//     waits in-kernel for the partials), one CTA per sequence: each warp merges
//     one row's partials and writes tokens / conf, a ballot over the B
//     confidences gives the commit count, and the committed K/V rows are
//     copied into the cache.
#include <cuda.h>
#include <math.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "lm_head.cuh"

namespace {

using namespace mars;

constexpr int kChunkVec = 1024;                 // 16-byte vectors per chunk (16 KB)
constexpr int kSlots = 12;                      // ring slots = consumer warps
constexpr int kThreads = 32 * (kSlots + 1);     // + one producer warp
constexpr int kRingBytes = kSlots * kChunkVec * 16;
constexpr int kGroup = 4;                       // vectors per lane per step
constexpr int kSteps = kChunkVec / (32 * kGroup);

struct RowState {
  float m;   // running max (-inf when empty)
  int idx;   // smallest index holding m
  float s;   // sum of exp(x - m)
  float m2;  // second largest value, counting a repeat of m (-inf when none); margin gate only
};

struct __align__(16) Partial {
  float m;
  int idx;
  float s;
  float m2;
};

__device__ __forceinline__ RowState empty_state() { return RowState{-INFINITY, 0x7fffffff, 0.f, -INFINITY}; }

// Merge b into a: the larger max wins, equal maxima keep the lower index; the
// runner-up is the larger of the smaller max and the two runners-up.
__device__ __forceinline__ void merge(RowState& a, const RowState& b) {
  if (b.m == -INFINITY) return;
  if (a.m == -INFINITY) {
    a = b;
    return;
  }
  a.m2 = fmaxf(fminf(a.m, b.m), fmaxf(a.m2, b.m2));
  if (b.m > a.m) {
    a.s = a.s * fast_exp2((a.m - b.m) * kLog2e) + b.s;
    a.m = b.m;
    a.idx = b.idx;
  } else if (b.m < a.m) {
    a.s += b.s * fast_exp2((b.m - a.m) * kLog2e);
  } else {
    a.s += b.s;
    a.idx = min(a.idx, b.idx);
  }
}

__device__ __forceinline__ RowState shfl_state(const RowState& a, int lane_mask) {
  RowState b;
  b.m = __shfl_xor_sync(0xffffffffu, a.m, lane_mask);
  b.idx = __shfl_xor_sync(0xffffffffu, a.idx, lane_mask);
  b.s = __shfl_xor_sync(0xffffffffu, a.s, lane_mask);
  b.m2 = __shfl_xor_sync(0xffffffffu, a.m2, lane_mask);
  return b;
}

__device__ __forceinline__ RowState warp_reduce(RowState st) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) merge(st, shfl_state(st, o));
  return st;
}

// Add one scalar element (index order not assumed).
__device__ __forceinline__ void add_scalar(RowState& st, float x, int idx) {
  merge(st, RowState{x, idx, 1.f, -INFINITY});
}

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hmax2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t bmin2(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hmin2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
// Top two of the values seen so far in each half of a packed bf16 pair (t1 >= t2).
__device__ __forceinline__ void top2_pair(uint32_t& t1, uint32_t& t2, uint32_t w) {
  t2 = bmax2(t2, bmin2(t1, w));
  t1 = bmax2(t1, w);
}

// acc2 (+)= exp2(x * log2e + mneg) for the two bf16 values packed in w, using
// packed fp32x2 FMA / ADD so one instruction serves both halves.
__device__ __forceinline__ void exp2_accumulate_pair(uint64_t& acc2, uint32_t w, float mneg) {
  const float lo = bf16lo_to_f32(w), hi = bf16hi_to_f32(w);
  float t0, t1;
  asm("{\n .reg .b64 x, c, b, t;\n mov.b64 x, {%2, %3};\n mov.b64 c, {%4, %4};\n mov.b64 b, {%5, %5};\n"
      " fma.rn.f32x2 t, x, c, b;\n mov.b64 {%0, %1}, t;\n}\n"
      : "=f"(t0), "=f"(t1)
      : "f"(lo), "f"(hi), "f"(kLog2e), "f"(mneg));
  const float e0 = fast_exp2(t0), e1 = fast_exp2(t1);
  asm("{\n .reg .b64 e;\n mov.b64 e, {%1, %2};\n add.rn.f32x2 %0, %0, e;\n}\n" : "+l"(acc2) : "f"(e0), "f"(e1));
}
__device__ __forceinline__ uint64_t pair_scale(uint64_t acc2, float f) {
  uint64_t r;
  asm("{\n .reg .b64 c;\n mov.b64 c, {%2, %2};\n mul.rn.f32x2 %0, %1, c;\n}\n" : "=l"(r) : "l"(acc2), "f"(f));
  return r;
}
__device__ __forceinline__ float pair_sum(uint64_t acc2) {
  return __uint_as_float(static_cast<uint32_t>(acc2)) + __uint_as_float(static_cast<uint32_t>(acc2 >> 32));
}

struct AcceptArgs {
  const uint16_t* logits;
  int batch, B, V;
  float tau;
  const uint16_t* k_new;
  const uint16_t* v_new;
  uint16_t* k_cache;
  uint16_t* v_cache;
  int32_t* cache_len;
  int Hkv, D, cap;
  int32_t* tokens;
  float* conf;
  int32_t* n_commit;
  int32_t* status;
  int margin;           // 1: conf = p1 - p2 (margin gate); 0: conf = p1
  int batch_min;        // 1: every sequence commits the batch minimum of the counts
  int deferred;         // 1: deferred-KV sampler: the cursor advances by the previous count, no K/V copy
  Partial* partials;    // [rows][chunks]
  int32_t* counts;      // [batch] per-sequence counts (batch-minimum mode), after the partials
  int chunks;           // chunks per row
  int items;            // rows * chunks
};

// Chunk k of row r: aligned vectors [v0, v1) plus the row's scalar head/tail bounds.
struct Chunk {
  const uint16_t* row;
  int head, tail0, v0, v1;
};

__device__ __forceinline__ Chunk chunk_of(const AcceptArgs& a, int r, int k) {
  Chunk c;
  c.row = a.logits + static_cast<size_t>(r) * a.V;
  // Elements [0, head) and [tail0, V) are not 16-byte aligned and are read as scalars.
  c.head = min(static_cast<int>(((16u - (reinterpret_cast<uintptr_t>(c.row) & 15u)) & 15u) >> 1), a.V);
  const int nvec = (a.V - c.head) >> 3;
  c.tail0 = c.head + 8 * nvec;
  c.v0 = min(nvec, k * kChunkVec);
  c.v1 = min(nvec, c.v0 + kChunkVec);
  return c;
}

// Second launch: one CTA per sequence b, one warp per proposal position i.
// Warp i merges the chunk partials of row (b, i) and writes tokens / conf;
// then the leading positions with conf >= tau are counted from a ballot (at
// least one), and the committed K/V rows are copied into the cache.  The
// partials, cache_len and (up to kPrefetch vectors per thread of) the B
// candidate K/V rows are all requested up front, so the launch costs about
// one memory round trip plus the stores.
constexpr int kPrefetch = 4;

__global__ void __launch_bounds__(32 * 16) accept_finish_kernel(const AcceptArgs a) {
  __shared__ float s_conf[16];
  __shared__ int s_n;
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int vec_per_row = a.D >> 3;
  const int per_pos = a.Hkv * vec_per_row;
  const int cand = a.deferred ? 0 : a.B * per_pos;  // candidate 16-byte vectors of K (and of V)
  const int len0 = __ldg(a.cache_len + b);
  // deferred-KV mode: the rows committed by the previous step, which this step's
  // decode attention has just written at the cursor
  const int pend = a.deferred ? a.n_commit[b] : 0;
  uint4 kpre[kPrefetch], vpre[kPrefetch];
#pragma unroll
  for (int u = 0; u < kPrefetch; ++u) {
    const int e = threadIdx.x + u * blockDim.x;
    if (e < cand) {
      const size_t src = (static_cast<size_t>(b) * a.B * per_pos + e) * 8;  // rows of [B, Hkv, D] are contiguous
      kpre[u] = *reinterpret_cast<const uint4*>(a.k_new + src);
      vpre[u] = *reinterpret_cast<const uint4*>(a.v_new + src);
    }
  }
  griddep_wait();  // the streaming launch's partials are complete and visible from here on
  griddep_launch_dependents();  // the next kernel (a decode step) may start its set-up
  {
    const int r = b * a.B + warp;
    RowState mg = empty_state();
    for (int s = lane; s < a.chunks; s += 32) {
      const float4 p = __ldcg(reinterpret_cast<const float4*>(a.partials + static_cast<size_t>(r) * a.chunks + s));
      merge(mg, RowState{p.x, __float_as_int(p.y), p.z, p.w});
    }
    const RowState st = warp_reduce(mg);
    if (lane == 0) {
      // p1 = 1 / s; margin gate: p1 - p2 = (1 - exp(m2 - m)) / s (0 on a tie, p1 if no runner-up)
      const float conf = a.margin ? (1.0f - fast_exp2((st.m2 - st.m) * kLog2e)) / st.s : 1.0f / st.s;
      a.tokens[r] = st.idx;
      a.conf[r] = conf;
      s_conf[warp] = conf;
    }
  }
  __syncthreads();
  if (warp == 0) {
    const bool pass = lane < a.B && s_conf[min(lane, a.B - 1)] >= a.tau;
    const uint32_t ok = __ballot_sync(0xffffffffu, pass);
    if (a.batch_min) {
      // the batch-minimum launch that follows commits and appends
      if (lane == 0) a.counts[b] = max(min(__ffs(~ok) - 1, a.B), 1);
      return;
    }
    if (lane == 0) {
      int n = max(min(__ffs(~ok) - 1, a.B), 1);
      const int base = len0 + pend;  // the cursor once the pending rows count
      const bool bad = len0 < 0 || pend < 0 || pend > a.B || base > a.cap;
      if (bad || base + n > a.cap) {
        set_status(a.status, MARS_DEV_CAPACITY);
        n = 0;
      }
      s_n = a.deferred ? 0 : n;
      a.n_commit[b] = n;
      a.cache_len[b] = bad ? len0 : base + (a.deferred ? 0 : n);
    }
  }
  if (a.batch_min) return;
  __syncthreads();
  // ---- block-level KV append of the committed rows: candidate vector e is
  // (position i, head g, chunk c) with e = (i * Hkv + g) * vec_per_row + c
  const int n = s_n;
  auto store = [&](int e, const uint4& kv, const uint4& vv) {
    const int i = e / per_pos;
    const int g = (e / vec_per_row) % a.Hkv;
    const int c = e % vec_per_row;
    const size_t dst = ((static_cast<size_t>(b) * a.Hkv + g) * a.cap + len0 + i) * a.D + 8 * c;
    *reinterpret_cast<uint4*>(a.k_cache + dst) = kv;
    *reinterpret_cast<uint4*>(a.v_cache + dst) = vv;
  };
#pragma unroll
  for (int u = 0; u < kPrefetch; ++u) {
    const int e = threadIdx.x + u * blockDim.x;
    if (e < n * per_pos) store(e, kpre[u], vpre[u]);
  }
  for (int e = threadIdx.x + kPrefetch * blockDim.x; e < n * per_pos; e += blockDim.x) {
    const size_t src = (static_cast<size_t>(b) * a.B * per_pos + e) * 8;
    store(e, *reinterpret_cast<const uint4*>(a.k_new + src), *reinterpret_cast<const uint4*>(a.v_new + src));
  }
}

template <bool kMargin>
__global__ void __launch_bounds__(kThreads, 1) accept_kernel(const AcceptArgs a) {
  extern __shared__ __align__(128) uint4 ring[];  // [kSlots][kChunkVec]
  __shared__ __align__(8) uint64_t full[kSlots], empty[kSlots];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  // Launched as a programmatic dependent of whatever precedes it in the stream: the
  // set-up above overlaps that kernel, and nothing global is read before it has
  // completed.  Only then may the finish launch start: it prefetches the candidate
  // K/V rows, which that kernel may have written, before it waits for this one.
  griddep_wait();
  griddep_launch_dependents();  // the finish launch may start prefetching beside us

  if (warp == kSlots) {
    // ================= producer: the CTA's chunks, in order, through the ring
    if (lane == 0) {
      int j = 0;  // CTA-local chunk sequence number; slot = j % kSlots
      for (int item = blockIdx.x; item < a.items; item += gridDim.x, ++j) {
        const int slot = j % kSlots;
        if (j >= kSlots && !mbar_wait(&empty[slot], ((j / kSlots) - 1) & 1)) {
          set_status(a.status, MARS_DEV_TIMEOUT);
          return;
        }
        const Chunk c = chunk_of(a, item / a.chunks, item % a.chunks);
        const uint32_t bytes = static_cast<uint32_t>(c.v1 - c.v0) * 16u;
        mbar_arrive_expect_tx(&full[slot], bytes);  // bytes == 0 completes the phase at once
        if (bytes > 0)
          bulk_g2s(smem_u32(ring + slot * kChunkVec), reinterpret_cast<const uint4*>(c.row + c.head) + c.v0, bytes,
                   &full[slot]);
      }
    }
    return;
  }

  // ================= consumer warp `warp`: chunks j = warp, warp + kSlots, ...
  const uint4 kNegInf = make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
  const uint4* buf = ring + warp * kChunkVec;
  int j = warp;
  for (int item = blockIdx.x + warp * gridDim.x; item < a.items; item += kSlots * gridDim.x, j += kSlots) {
    const int r = item / a.chunks, k = item % a.chunks;
    const Chunk c = chunk_of(a, r, k);
    if (!mbar_wait(&full[warp], (j / kSlots) & 1)) {
      if (lane == 0) set_status(a.status, MARS_DEV_TIMEOUT);
      return;
    }
    const int n = c.v1 - c.v0;

    // ---- the chunk: lane l reads vectors l + 32 * (kGroup * step + u), index order per lane
    float m = -INFINITY, mneg = 0.f;
    uint64_t acc2 = 0;
    int best_step = -1;
    uint4 best[kGroup];
    uint32_t t1 = 0xff80ff80u, t2 = 0xff80ff80u;  // margin gate: per-half top two (bf16 -inf)
#pragma unroll 2
    for (int step = 0; step < kSteps; ++step) {
      uint4 w[kGroup];
#pragma unroll
      for (int u = 0; u < kGroup; ++u) {
        const int vi = lane + 32 * (kGroup * step + u);
        w[u] = vi < n ? buf[vi] : kNegInf;
      }
      if (kMargin) {
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
          top2_pair(t1, t2, w[u].x);
          top2_pair(t1, t2, w[u].y);
          top2_pair(t1, t2, w[u].z);
          top2_pair(t1, t2, w[u].w);
        }
      }
      uint32_t mx = bmax2(bmax2(w[0].x, w[0].y), bmax2(w[0].z, w[0].w));
#pragma unroll
      for (int u = 1; u < kGroup; ++u) mx = bmax2(mx, bmax2(bmax2(w[u].x, w[u].y), bmax2(w[u].z, w[u].w)));
      const float gmax = fmaxf(bf16lo_to_f32(mx), bf16hi_to_f32(mx));
      if (gmax > m) {
        acc2 = pair_scale(acc2, fast_exp2((m - gmax) * kLog2e));  // exp2(-inf) = 0 on the first group
        m = gmax;
        mneg = -gmax * kLog2e;
        best_step = step;
#pragma unroll
        for (int u = 0; u < kGroup; ++u) best[u] = w[u];
      }
#pragma unroll
      for (int u = 0; u < kGroup; ++u) {
        exp2_accumulate_pair(acc2, w[u].x, mneg);
        exp2_accumulate_pair(acc2, w[u].y, mneg);
        exp2_accumulate_pair(acc2, w[u].z, mneg);
        exp2_accumulate_pair(acc2, w[u].w, mneg);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[warp]);  // the slot is free again

    RowState st = empty_state();
    if (best_step >= 0) {
      int found = 0x7fffffff;
#pragma unroll
      for (int u = kGroup - 1; u >= 0; --u) {
        const uint32_t ws[4] = {best[u].x, best[u].y, best[u].z, best[u].w};
#pragma unroll
        for (int e = 7; e >= 0; --e) {
          const float x = (e & 1) ? bf16hi_to_f32(ws[e >> 1]) : bf16lo_to_f32(ws[e >> 1]);
          if (x == m) found = c.head + 8 * (c.v0 + lane + 32 * (kGroup * best_step + u)) + e;
        }
      }
      // runner-up of the lane: the smaller half-maximum or either half's second
      const float m2 = kMargin ? fmaxf(fminf(bf16lo_to_f32(t1), bf16hi_to_f32(t1)),
                                       fmaxf(bf16lo_to_f32(t2), bf16hi_to_f32(t2)))
                               : -INFINITY;
      st = RowState{m, found, pair_sum(acc2), m2};
    }
    // ---- unaligned head (first chunk) and tail (last chunk): at most 7 + 7 elements
    if (k == 0 && lane < c.head) add_scalar(st, bf16lo_to_f32(c.row[lane]), lane);
    if (k == a.chunks - 1 && c.tail0 + lane < a.V) add_scalar(st, bf16lo_to_f32(c.row[c.tail0 + lane]), c.tail0 + lane);
    st = warp_reduce(st);
    if (lane == 0) a.partials[static_cast<size_t>(r) * a.chunks + k] = Partial{st.m, st.idx, st.s, st.m2};
  }

}

inline int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// Chunks per row of V logits (a row's aligned part has at most ceil(V/8) vectors).
inline int chunks_for(int V) { return max(1, ceil_div(ceil_div(V, 8), kChunkVec)); }

// Batch-minimum mode (the paper's original sampler: the block-level cache of a
// batch advances at its minimum acceptance): one CTA per sequence commits
// n = min over the batch of the per-sequence counts and appends n rows.
__global__ void __launch_bounds__(256) accept_batchmin_kernel(const AcceptArgs a) {
  __shared__ int s_min[8];
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int len0 = __ldg(a.cache_len + b);
  const int pend = a.deferred ? a.n_commit[b] : 0;  // deferred-KV mode: the previous step's count
  griddep_wait();  // the per-sequence counts are complete and visible from here on
  int m = a.B;
  for (int t = threadIdx.x; t < a.batch; t += blockDim.x) m = min(m, __ldcg(a.counts + t));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = min(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) s_min[warp] = m;
  __syncthreads();
  int n = s_min[0];
  for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) n = min(n, s_min[w]);
  const int base = len0 + pend;
  const bool bad = len0 < 0 || pend < 0 || pend > a.B || base > a.cap;
  if (bad || base + n > a.cap) {
    if (threadIdx.x == 0) {
      set_status(a.status, MARS_DEV_CAPACITY);
      a.n_commit[b] = 0;
      if (!bad) a.cache_len[b] = base;
    }
    return;
  }
  if (threadIdx.x == 0) {
    a.n_commit[b] = n;
    a.cache_len[b] = base + (a.deferred ? 0 : n);
  }
  if (a.deferred) return;
  const int vec_per_row = a.D >> 3;
  const int per_pos = a.Hkv * vec_per_row;
  for (int e = threadIdx.x; e < n * per_pos; e += blockDim.x) {
    const size_t src = (static_cast<size_t>(b) * a.B * per_pos + e) * 8;
    const int i = e / per_pos, g = (e / vec_per_row) % a.Hkv, c = e % vec_per_row;
    const size_t dst = ((static_cast<size_t>(b) * a.Hkv + g) * a.cap + len0 + i) * a.D + 8 * c;
    *reinterpret_cast<uint4*>(a.k_cache + dst) = *reinterpret_cast<const uint4*>(a.k_new + src);
    *reinterpret_cast<uint4*>(a.v_cache + dst) = *reinterpret_cast<const uint4*>(a.v_new + src);
  }
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace: one Partial per (row, chunk).
inline size_t partial_bytes(int batch, int B, int V) {
  return align_up(static_cast<size_t>(batch) * B * chunks_for(V) * sizeof(Partial), 256);
}
// Workspace: the partials, then one count per sequence (batch-minimum mode).
inline size_t ws_bytes(int batch, int B, int V) {
  return partial_bytes(batch, B, V) + align_up(static_cast<size_t>(batch) * sizeof(int32_t), 256);
}

int configure_kernel() {
  static int done[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MARS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(accept_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(accept_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes);
    if (e != cudaSuccess) return mars_host::cuda_fail(e);
    done[dev] = 1;
  }
  return MARS_OK;
}

int launch_finish(AcceptArgs& a, cudaStream_t stream);

int launch(AcceptArgs& a, cudaStream_t stream) {
  const int rc = configure_kernel();
  if (rc != MARS_OK) return rc;
  a.chunks = chunks_for(a.V);
  a.items = a.batch * a.B * a.chunks;
  const int grid = std::min(a.items, mars_host::num_sms());
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kRingBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = a.margin ? cudaLaunchKernelEx(&cfg, accept_kernel<true>, a)
                                   : cudaLaunchKernelEx(&cfg, accept_kernel<false>, a);
    if (e != cudaSuccess) return mars_host::cuda_fail(e);
  }
  return launch_finish(a, stream);
}

// The finish launch (and, in batch-minimum mode, the minimum launch): one CTA per
// sequence.  It overlaps its start-up and prefetch with the launch that produces
// the partials (programmatic dependent launch) and waits for them in-kernel.
int launch_finish(AcceptArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.batch, 1, 1);
  cfg.blockDim = dim3(32 * a.B, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, accept_finish_kernel, a);
  if (e != cudaSuccess || !a.batch_min) return e == cudaSuccess ? MARS_OK : mars_host::cuda_fail(e);
  cfg.gridDim = dim3(a.batch, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  e = cudaLaunchKernelEx(&cfg, accept_batchmin_kernel, a);
  return e == cudaSuccess ? MARS_OK : mars_host::cuda_fail(e);
}

// Host-side argument checks shared by both entry points.
int check_args(const uint16_t* logits, int batch, int B, int V, float tau, const uint16_t* k_new,
               const uint16_t* v_new, const uint16_t* k_cache, const uint16_t* v_cache, const int32_t* cache_len,
               int Hkv, int D, int cap, const int32_t* tokens, const float* conf, const int32_t* n_commit,
               const int32_t* status, bool with_kv = true) {
  using mars_host::aligned16;
  using mars_host::aligned2;
  using mars_host::aligned4;
  MARS_HOST_CHECK(batch > 0 && B > 0 && B <= 16 && V > 0 && cap > 0, MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(static_cast<long long>(batch) * B * chunks_for(V) < (1LL << 31), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(!isnan(tau), MARS_ERR_INVALID_ARG);
  if (with_kv) {
    MARS_HOST_CHECK(Hkv > 0 && D > 0 && D % 8 == 0 && D <= 256, MARS_ERR_INVALID_ARG);
    const void* vec16[] = {k_new, v_new, k_cache, v_cache};
    for (const void* p : vec16) MARS_HOST_CHECK(p != nullptr && aligned16(p), MARS_ERR_INVALID_ARG);
  }
  const void* word4[] = {cache_len, tokens, conf, n_commit};
  for (const void* p : word4) MARS_HOST_CHECK(p != nullptr && aligned4(p), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(logits != nullptr && aligned2(logits), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(status == nullptr || aligned4(status), MARS_ERR_INVALID_ARG);
  return MARS_OK;
}

AcceptArgs make_args(const uint16_t* logits, int batch, int B, int V, float tau, const uint16_t* k_new,
                     const uint16_t* v_new, uint16_t* k_cache, uint16_t* v_cache, int32_t* cache_len, int Hkv, int D,
                     int cap, int32_t* tokens, float* conf, int32_t* n_commit, int32_t* status) {
  AcceptArgs a;
  a.logits = logits;
  a.batch = batch;
  a.B = B;
  a.V = V;
  a.tau = tau;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.cache_len = cache_len;
  a.Hkv = Hkv;
  a.D = D;
  a.cap = cap;
  a.tokens = tokens;
  a.conf = conf;
  a.n_commit = n_commit;
  a.status = status;
  a.margin = 0;
  a.batch_min = 0;
  a.deferred = 0;
  a.partials = nullptr;
  a.counts = nullptr;
  a.chunks = a.items = 0;
  return a;
}

}  // namespace

extern "C" size_t mars_accept_workspace_size(int batch, int B, int V) {
  if (batch <= 0 || B <= 0 || V <= 0) return 0;
  return ws_bytes(batch, B, V);
}

extern "C" int mars_accept_ex(const uint16_t* logits, int batch, int B, int V, float tau, int flags,
                              const uint16_t* k_new, const uint16_t* v_new, uint16_t* k_cache, uint16_t* v_cache,
                              int32_t* cache_len, int Hkv, int D, int cap, int32_t* tokens, float* conf,
                              int32_t* n_commit, int32_t* status, void* workspace, size_t workspace_bytes,
                              void* stream) {
  MARS_HOST_CHECK((flags & ~(MARS_ACCEPT_MARGIN | MARS_ACCEPT_BATCH_MIN | MARS_ACCEPT_DEFERRED)) == 0,
                  MARS_ERR_INVALID_ARG);
  const bool deferred = (flags & MARS_ACCEPT_DEFERRED) != 0;
  int rc = check_args(logits, batch, B, V, tau, k_new, v_new, k_cache, v_cache, cache_len, Hkv, D, cap, tokens,
                      conf, n_commit, status, !deferred);
  if (rc != MARS_OK) return rc;
  MARS_HOST_CHECK(workspace != nullptr && mars_host::aligned16(workspace), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(workspace_bytes >= ws_bytes(batch, B, V), MARS_ERR_WORKSPACE_TOO_SMALL);
  rc = mars_host::check_device();
  if (rc != MARS_OK) return rc;

  AcceptArgs a = make_args(logits, batch, B, V, tau, k_new, v_new, k_cache, v_cache, cache_len, Hkv, D, cap, tokens,
                           conf, n_commit, status);
  a.margin = (flags & MARS_ACCEPT_MARGIN) ? 1 : 0;
  a.batch_min = (flags & MARS_ACCEPT_BATCH_MIN) ? 1 : 0;
  a.deferred = deferred ? 1 : 0;
  a.partials = static_cast<Partial*>(workspace);
  a.counts = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + partial_bytes(batch, B, V));
  return launch(a, static_cast<cudaStream_t>(stream));
}

extern "C" int mars_accept(const uint16_t* logits, int batch, int B, int V, float tau, const uint16_t* k_new,
                           const uint16_t* v_new, uint16_t* k_cache, uint16_t* v_cache, int32_t* cache_len, int Hkv,
                           int D, int cap, int32_t* tokens, float* conf, int32_t* n_commit, int32_t* status,
                           void* workspace, size_t workspace_bytes, void* stream) {
  return mars_accept_ex(logits, batch, B, V, tau, 0, k_new, v_new, k_cache, v_cache, cache_len, Hkv, D, cap, tokens,
                        conf, n_commit, status, workspace, workspace_bytes, stream);
}

extern "C" int mars_accept_margin(const uint16_t* logits, int batch, int B, int V, float tau, const uint16_t* k_new,
                                  const uint16_t* v_new, uint16_t* k_cache, uint16_t* v_cache, int32_t* cache_len,
                                  int Hkv, int D, int cap, int32_t* tokens, float* conf, int32_t* n_commit,
                                  int32_t* status, void* workspace, size_t workspace_bytes, void* stream) {
  return mars_accept_ex(logits, batch, B, V, tau, MARS_ACCEPT_MARGIN, k_new, v_new, k_cache, v_cache, cache_len, Hkv,
                        D, cap, tokens, conf, n_commit, status, workspace, workspace_bytes, stream);
}

// ============================================================================
// mars_accept_noalloc: the same computation with library-owned scratch.
//
// Some callers cannot hand the library a workspace: a plugin that only sees
// the input and output buffers its host framework gives it, or a serving loop
// running under a fixed device-memory budget, where cudaMalloc could fail in
// the middle of decoding and would synchronise the whole device.  This entry
// point allocates nothing.  Its scratch is a file-scope device array of
// kNoAllocScratchBytes that every GPU loading this library keeps until the
// process exits.
//
// The array holds only the per-chunk partial results of the current call
// (batch * B * ceil(V / 8192) of them, at most 65536); nothing in it has to
// start at zero, and each call overwrites what it reads.
// ============================================================================
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
constexpr size_t kNoAllocPartialSlots = kNoAllocScratchBytes / sizeof(Partial);
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) uint8_t g_accept_scratch[kNoAllocScratchBytes];

// The array's device address, resolved once per (device, CUDA context): a new
// context on the same device (after cudaDeviceReset, say) reloads the module,
// possibly at another address, so the cache is keyed on the context's id too.
struct ScratchAddr {
  unsigned long long ctx_id;
  void* ptr;
};
ScratchAddr g_noalloc_scratch[kNoAllocMaxDevices];
std::mutex g_noalloc_mu;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Id of the calling thread's current CUDA context (0 if it cannot be read).
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_accept_scratch in the current device's context.  The first
// call in a context resolves it with that device current (in host code the
// array's name is only a host-side stand-in, not a device address).  That look-up
// is not a stream operation, so it is refused while `stream` is being captured.
int noalloc_scratch(cudaStream_t stream, char** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MARS_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return MARS_ERR_UNSUPPORTED_DEVICE;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  ScratchAddr& slot = g_noalloc_scratch[dev];
  if (slot.ptr == nullptr || slot.ctx_id != ctx || ctx == 0) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const cudaError_t ce = cudaStreamIsCapturing(stream, &cs);
    if (ce != cudaSuccess) return mars_host::cuda_fail(ce);
    if (cs != cudaStreamCaptureStatusNone) return MARS_ERR_SCRATCH_NOT_READY;
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_accept_scratch);
    if (e != cudaSuccess || p == nullptr) return mars_host::cuda_fail(e);
    slot.ptr = p;
    slot.ctx_id = ctx;
  }
  *out = static_cast<char*>(slot.ptr);
  return MARS_OK;
}

}  // namespace

extern "C" int mars_accept_noalloc(const uint16_t* logits, int batch, int B, int V, float tau,
                                   const uint16_t* k_new, const uint16_t* v_new, uint16_t* k_cache,
                                   uint16_t* v_cache, int32_t* cache_len, int Hkv, int D, int cap, int32_t* tokens,
                                   float* conf, int32_t* n_commit, int32_t* status, void* stream) {
  int rc = check_args(logits, batch, B, V, tau, k_new, v_new, k_cache, v_cache, cache_len, Hkv, D, cap, tokens,
                      conf, n_commit, status);
  if (rc != MARS_OK) return rc;
  MARS_HOST_CHECK(static_cast<long long>(batch) * B * chunks_for(V) <= static_cast<long long>(kNoAllocPartialSlots),
                  MARS_ERR_SCRATCH_LIMIT);
  rc = mars_host::check_device();
  if (rc != MARS_OK) return rc;
  char* scratch = nullptr;
  rc = noalloc_scratch(static_cast<cudaStream_t>(stream), &scratch);
  if (rc != MARS_OK) return rc;

  AcceptArgs a = make_args(logits, batch, B, V, tau, k_new, v_new, k_cache, v_cache, cache_len, Hkv, D, cap, tokens,
                           conf, n_commit, status);
  a.partials = reinterpret_cast<Partial*>(scratch);
  return launch(a, static_cast<cudaStream_t>(stream));
}

// ============================================================================
// mars_lm_head_accept: the LM head fused with the acceptance step.  The head's
// kernel (lm_head.cu) reduces each row's logits tile by tile to one partial per
// vocabulary range; the finish launch above merges them, applies the commit
// rule and appends, exactly as for mars_accept.
// ============================================================================
extern "C" size_t mars_lm_head_accept_workspace_size(int batch, int B, int V) {
  if (batch <= 0 || B <= 0 || V <= 0) return 0;
  const int rows = batch * B;
  return align_up(static_cast<size_t>(rows) * mars_lm_head::splits_for(rows, V) * sizeof(Partial), 256);
}

extern "C" int mars_lm_head_accept(const uint16_t* hidden, const uint16_t* weight, int batch, int B, int K, int V,
                                   float tau, const uint16_t* k_new, const uint16_t* v_new, uint16_t* k_cache,
                                   uint16_t* v_cache, int32_t* cache_len, int Hkv, int D, int cap, int32_t* tokens,
                                   float* conf, int32_t* n_commit, int32_t* status, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  int rc = check_args(hidden, batch, B, V, tau, k_new, v_new, k_cache, v_cache, cache_len, Hkv, D, cap, tokens, conf,
                      n_commit, status);
  if (rc != MARS_OK) return rc;
  MARS_HOST_CHECK(K >= 64 && K % 64 == 0 && V < (1 << 30), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(mars_host::aligned16(hidden) && weight != nullptr && mars_host::aligned16(weight),
                  MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(workspace != nullptr && mars_host::aligned16(workspace), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(workspace_bytes >= mars_lm_head_accept_workspace_size(batch, B, V), MARS_ERR_WORKSPACE_TOO_SMALL);
  rc = mars_host::check_device();
  if (rc != MARS_OK) return rc;
  const int rows = batch * B;
  const int nsplit = mars_lm_head::splits_for(rows, V);
  rc = mars_lm_head::launch_partials(hidden, weight, rows, K, V, static_cast<float4*>(workspace), nsplit, status,
                                     static_cast<cudaStream_t>(stream));
  if (rc != MARS_OK) return rc;
  AcceptArgs a = make_args(hidden, batch, B, V, tau, k_new, v_new, k_cache, v_cache, cache_len, Hkv, D, cap, tokens,
                           conf, n_commit, status);
  a.partials = static_cast<Partial*>(workspace);
  a.chunks = nsplit;
  a.items = rows * nsplit;
  return launch_finish(a, static_cast<cudaStream_t>(stream));
}
