// accept.cu - mars_accept: top-1 probability, greedy token, left-to-right
// commit with threshold tau, and the block-level KV append, in one launch.
//
// Method: the authors' MARS blog post, "Inference: a knob, not a mode switch"
// (commit while the top-1 probability holds, stop at the first position below
// tau); "MARS: Enabling Autoregressive Models Multi-Token Generation",
// Sec. 3.1 gap (4) (strictly left to right) and its block-level KV cache
// contribution; the aitrends.kr summary (at least one token is accepted).
//
// Design (HBM-bound, one read of the logits):
//   grid = (splits, batch * B).  CTA (s, r) streams a contiguous slice of row
//   r with 16-byte loads, UNROLL of them in flight per thread, and keeps a
//   running (max, argmax, sum exp(x - max)) per thread.  The max of each
//   loaded batch is taken first on packed bf16, so the exponentials are taken
//   against a running max that rarely moves, and the argmax only needs a scan
//   when the batch max beats it.  Warp shuffles and shared memory reduce the
//   CTA; the partial goes to the workspace.  The last CTA of a row (an atomic
//   ticket, no waiting) merges the partials and writes tokens / conf; the last
//   row of a sequence computes n_commit and copies the committed K/V rows into
//   the cache.  Tickets are reset by their last user, so the counters are
//   zero again after every call (the partial slots are simply overwritten).
#include <math.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace {

using namespace mars;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;          // 16-byte loads in flight per thread
constexpr int kMinChunkVec = 256;   // smallest slice per CTA, in 16-byte vectors (4 KB)

struct RowState {
  float m;   // running max (-inf when empty)
  int idx;   // smallest index holding m
  float s;   // sum of exp(x - m)
};

struct __align__(16) Partial {
  float m;
  int idx;
  float s;
  int pad;
};

__device__ __forceinline__ RowState empty_state() { return RowState{-INFINITY, 0x7fffffff, 0.f}; }

// Merge b into a: the larger max wins, equal maxima keep the lower index.
__device__ __forceinline__ void merge(RowState& a, const RowState& b) {
  if (b.m == -INFINITY) return;
  if (a.m == -INFINITY) {
    a = b;
    return;
  }
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
  return b;
}

// Add one scalar element (index increasing is NOT assumed).
__device__ __forceinline__ void add_scalar(RowState& st, float x, int idx) {
  RowState one{x, idx, 1.f};
  merge(st, one);
}

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hmax2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ RowState block_reduce(RowState st, RowState* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) merge(st, shfl_state(st, o));
  if (lane == 0) red[warp] = st;
  __syncthreads();
  if (warp == 0) {
    st = lane < kWarps ? red[lane] : empty_state();
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) merge(st, shfl_state(st, o));
  }
  return st;  // valid in thread 0
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
  Partial* partials;    // [rows][splits]
  int32_t* row_ticket;  // [rows]
  int32_t* seq_ticket;  // [batch]
  int splits;
  int chunk_vec;        // vectors per CTA slice
};

__global__ void __launch_bounds__(kThreads) accept_kernel(const AcceptArgs a) {
  __shared__ RowState red[kWarps];
  __shared__ int flag;

  const int split = blockIdx.x;
  const int r = blockIdx.y;  // row = b * B + i
  const int tid = threadIdx.x;
  const uint16_t* row = a.logits + static_cast<size_t>(r) * a.V;

  // Elements [0, head) and [head + 8 * nvec, V) are not 16-byte aligned and are read as scalars.
  const int head = min(static_cast<int>(((16u - (reinterpret_cast<uintptr_t>(row) & 15u)) & 15u) >> 1), a.V);
  const int nvec = (a.V - head) >> 3;
  const int tail0 = head + 8 * nvec;
  const int v0 = split * a.chunk_vec;
  const int v1 = min(nvec, v0 + a.chunk_vec);

  RowState st = empty_state();
  // ---- vector body: thread-local indices increase monotonically
  {
    const uint4* vp = reinterpret_cast<const uint4*>(row + head);
    float m = -INFINITY, mneg = 0.f, s0 = 0.f, s1 = 0.f;
    int idx = 0x7fffffff;
    for (int base = v0 + tid; base < v1; base += kThreads * kUnroll) {
      uint4 w[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int vi = base + u * kThreads;
        w[u] = vi < v1 ? __ldcs(vp + vi) : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
      }
      uint32_t mx = bmax2(bmax2(w[0].x, w[0].y), bmax2(w[0].z, w[0].w));
#pragma unroll
      for (int u = 1; u < kUnroll; ++u) mx = bmax2(mx, bmax2(bmax2(w[u].x, w[u].y), bmax2(w[u].z, w[u].w)));
      const float gmax = fmaxf(bf16lo_to_f32(mx), bf16hi_to_f32(mx));
      if (gmax > m) {
        // first element equal to the new max, in index order
        int found = 0x7fffffff;
#pragma unroll
        for (int u = kUnroll - 1; u >= 0; --u) {
          const uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
          for (int e = 7; e >= 0; --e) {
            const float x = (e & 1) ? bf16hi_to_f32(ws[e >> 1]) : bf16lo_to_f32(ws[e >> 1]);
            if (x == gmax) found = head + 8 * (base + u * kThreads) + e;
          }
        }
        const float f = fast_exp2((m - gmax) * kLog2e);
        s0 *= f;
        s1 *= f;
        m = gmax;
        mneg = -gmax * kLog2e;
        idx = found;
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          s0 += fast_exp2(fmaf(bf16lo_to_f32(ws[h]), kLog2e, mneg));
          s1 += fast_exp2(fmaf(bf16hi_to_f32(ws[h]), kLog2e, mneg));
        }
      }
    }
    st.m = m;
    st.idx = idx;
    st.s = s0 + s1;
    if (m == -INFINITY) st = empty_state();
  }
  // ---- unaligned head (split 0) and tail (last split): at most 7 + 7 elements
  if (split == 0 && tid < head) add_scalar(st, bf16lo_to_f32(row[tid]), tid);
  if (split == a.splits - 1 && tail0 + tid < a.V) add_scalar(st, bf16lo_to_f32(row[tail0 + tid]), tail0 + tid);

  st = block_reduce(st, red);

  // ---- row finalisation: by the only CTA (splits == 1) or the last one to finish
  if (tid == 0) {
    int last = 1;
    if (a.splits > 1) {
      a.partials[static_cast<size_t>(r) * a.splits + split] = Partial{st.m, st.idx, st.s, 0};
      __threadfence();
      last = atomicAdd(&a.row_ticket[r], 1) == a.splits - 1;
      if (last) {
        __threadfence();
        st = empty_state();
        for (int s = 0; s < a.splits; ++s) {
          const float4 p = __ldcg(reinterpret_cast<const float4*>(a.partials + static_cast<size_t>(r) * a.splits + s));
          merge(st, RowState{p.x, __float_as_int(p.y), p.z});
        }
        a.row_ticket[r] = 0;
      }
    }
    int seq_last = 0;
    if (last) {
      a.tokens[r] = st.idx;
      a.conf[r] = 1.0f / st.s;
      __threadfence();
      const int b = r / a.B;
      seq_last = atomicAdd(&a.seq_ticket[b], 1) == a.B - 1;
      if (seq_last) __threadfence();
    }
    flag = seq_last;
  }
  __syncthreads();
  if (!flag) return;

  // ---- sequence finalisation: commit count and KV append
  __shared__ int s_n, s_len;
  const int b = r / a.B;
  if (tid == 0) {
    int n = 0;
    for (int i = 0; i < a.B; ++i) {
      if (__ldcg(a.conf + b * a.B + i) >= a.tau) ++n;
      else break;
    }
    n = max(n, 1);
    const int len = __ldcg(a.cache_len + b);
    if (len < 0 || len + n > a.cap) {
      set_status(a.status, MARS_DEV_CAPACITY);
      n = 0;
    }
    a.n_commit[b] = n;
    s_n = n;
    s_len = len;
    a.seq_ticket[b] = 0;
  }
  __syncthreads();
  const int n = s_n, len = s_len;
  const int vec_per_row = a.D >> 3;
  const int per_pos = a.Hkv * vec_per_row;
  const int total = n * per_pos;
  for (int e = tid; e < total; e += kThreads) {
    const int i = e / per_pos;
    const int g = (e / vec_per_row) % a.Hkv;
    const int c = e % vec_per_row;
    const size_t src = ((static_cast<size_t>(b) * a.B + i) * a.Hkv + g) * a.D + 8 * c;
    const size_t dst = ((static_cast<size_t>(b) * a.Hkv + g) * a.cap + len + i) * a.D + 8 * c;
    *reinterpret_cast<uint4*>(a.k_cache + dst) = *reinterpret_cast<const uint4*>(a.k_new + src);
    *reinterpret_cast<uint4*>(a.v_cache + dst) = *reinterpret_cast<const uint4*>(a.v_new + src);
  }
  if (tid == 0) a.cache_len[b] = len + n;
}

inline int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// Number of 16-byte vectors per row that a CTA slice can cover at most.
inline int max_splits_for(int V) { return max(1, ceil_div(ceil_div(V, 8), kMinChunkVec)); }

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
  size_t partials, row_ticket, seq_ticket, total;
};

inline WsLayout ws_layout(int batch, int B, int V) {
  const size_t rows = static_cast<size_t>(batch) * B;
  WsLayout l;
  l.partials = 0;
  l.row_ticket = align_up(rows * max_splits_for(V) * sizeof(Partial), 256);
  l.seq_ticket = align_up(l.row_ticket + rows * sizeof(int32_t), 256);
  l.total = align_up(l.seq_ticket + static_cast<size_t>(batch) * sizeof(int32_t), 256);
  return l;
}

}  // namespace

extern "C" size_t mars_accept_workspace_size(int batch, int B, int V) {
  if (batch <= 0 || B <= 0 || V <= 0) return 0;
  return ws_layout(batch, B, V).total;
}

extern "C" int mars_accept(const uint16_t* logits, int batch, int B, int V, float tau, const uint16_t* k_new,
                           const uint16_t* v_new, uint16_t* k_cache, uint16_t* v_cache, int32_t* cache_len, int Hkv,
                           int D, int cap, int32_t* tokens, float* conf, int32_t* n_commit, int32_t* status,
                           void* workspace, size_t workspace_bytes, void* stream) {
  using mars_host::aligned16;
  using mars_host::aligned2;
  using mars_host::aligned4;
  MARS_HOST_CHECK(batch > 0 && B > 0 && B <= 16 && V > 0 && Hkv > 0 && D > 0 && D % 8 == 0 && D <= 256 && cap > 0,
                  MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(static_cast<long long>(batch) * B <= 65535, MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(!isnan(tau), MARS_ERR_INVALID_ARG);
  const void* vec16[] = {k_new, v_new, k_cache, v_cache, workspace};
  for (const void* p : vec16) MARS_HOST_CHECK(p != nullptr && aligned16(p), MARS_ERR_INVALID_ARG);
  const void* word4[] = {cache_len, tokens, conf, n_commit};
  for (const void* p : word4) MARS_HOST_CHECK(p != nullptr && aligned4(p), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(logits != nullptr && aligned2(logits), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(status == nullptr || aligned4(status), MARS_ERR_INVALID_ARG);
  const WsLayout l = ws_layout(batch, B, V);
  MARS_HOST_CHECK(workspace_bytes >= l.total, MARS_ERR_WORKSPACE_TOO_SMALL);
  int rc = mars_host::check_device();
  if (rc != MARS_OK) return rc;

  const int rows = batch * B;
  const int nvec_max = ceil_div(V, 8);
  const int target_ctas = 16 * mars_host::num_sms();
  int splits = std::min(max_splits_for(V), std::max(1, ceil_div(target_ctas, rows)));
  const int chunk_vec = ceil_div(nvec_max, splits);
  splits = ceil_div(nvec_max, chunk_vec);

  char* ws = static_cast<char*>(workspace);
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
  a.partials = reinterpret_cast<Partial*>(ws + l.partials);
  a.row_ticket = reinterpret_cast<int32_t*>(ws + l.row_ticket);
  a.seq_ticket = reinterpret_cast<int32_t*>(ws + l.seq_ticket);
  a.splits = splits;
  a.chunk_vec = chunk_vec;
  accept_kernel<<<dim3(splits, rows), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? MARS_OK : MARS_ERR_CUDA;
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
// Layout of the array (fixed, so the counters never share bytes with partial
// results of an earlier call of another shape):
//   [0, 16 KB)   per-row completion counters   (batch * B <= 4096)
//   [16, 32 KB)  per-sequence completion counters (batch <= 4096)
//   [32 KB, 1 MB) per-slice partial results; the number of vocabulary slices
//                is reduced when batch * B * slices would not fit.
// The counters are zeroed once, when the array is set up on a device, and
// every call returns them to zero.
// ============================================================================
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
constexpr int kNoAllocMaxRows = 4096;
constexpr int kNoAllocMaxBatch = 4096;
constexpr size_t kNoAllocRowTicketOff = 0;
constexpr size_t kNoAllocSeqTicketOff = kNoAllocRowTicketOff + sizeof(int32_t) * kNoAllocMaxRows;
constexpr size_t kNoAllocPartialOff = kNoAllocSeqTicketOff + sizeof(int32_t) * kNoAllocMaxBatch;
constexpr size_t kNoAllocPartialSlots = (kNoAllocScratchBytes - kNoAllocPartialOff) / sizeof(Partial);
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) uint8_t g_accept_scratch[kNoAllocScratchBytes];

void* g_noalloc_scratch[kNoAllocMaxDevices];
std::mutex g_noalloc_mu;

// Device address of g_accept_scratch on the current device.  The first call on
// a device resolves the address (in host code the array's name is only a
// host-side stand-in) and zeroes the counters, with that device current.
int noalloc_scratch(char** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MARS_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return MARS_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_scratch[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess || p == nullptr) return MARS_ERR_CUDA;
    if (cudaMemset(p, 0, kNoAllocPartialOff) != cudaSuccess) return MARS_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return MARS_ERR_CUDA;
    g_noalloc_scratch[dev] = p;
  }
  *out = static_cast<char*>(g_noalloc_scratch[dev]);
  return MARS_OK;
}

}  // namespace

extern "C" int mars_accept_noalloc(const uint16_t* logits, int batch, int B, int V, float tau,
                                   const uint16_t* k_new, const uint16_t* v_new, uint16_t* k_cache,
                                   uint16_t* v_cache, int32_t* cache_len, int Hkv, int D, int cap, int32_t* tokens,
                                   float* conf, int32_t* n_commit, int32_t* status, void* stream) {
  using mars_host::aligned16;
  using mars_host::aligned2;
  using mars_host::aligned4;
  MARS_HOST_CHECK(batch > 0 && B > 0 && B <= 16 && V > 0 && Hkv > 0 && D > 0 && D % 8 == 0 && D <= 256 && cap > 0,
                  MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(!isnan(tau), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(batch <= kNoAllocMaxBatch && static_cast<long long>(batch) * B <= kNoAllocMaxRows,
                  MARS_ERR_SCRATCH_LIMIT);
  const void* vec16[] = {k_new, v_new, k_cache, v_cache};
  for (const void* p : vec16) MARS_HOST_CHECK(p != nullptr && aligned16(p), MARS_ERR_INVALID_ARG);
  const void* word4[] = {cache_len, tokens, conf, n_commit};
  for (const void* p : word4) MARS_HOST_CHECK(p != nullptr && aligned4(p), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(logits != nullptr && aligned2(logits), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(status == nullptr || aligned4(status), MARS_ERR_INVALID_ARG);
  int rc = mars_host::check_device();
  if (rc != MARS_OK) return rc;
  char* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc != MARS_OK) return rc;

  const int rows = batch * B;
  const int nvec_max = ceil_div(V, 8);
  const int target_ctas = 16 * mars_host::num_sms();
  int splits = std::min(max_splits_for(V), std::max(1, ceil_div(target_ctas, rows)));
  splits = std::max(1, std::min(splits, static_cast<int>(kNoAllocPartialSlots / rows)));
  const int chunk_vec = ceil_div(nvec_max, splits);
  splits = ceil_div(nvec_max, chunk_vec);

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
  a.partials = reinterpret_cast<Partial*>(scratch + kNoAllocPartialOff);
  a.row_ticket = reinterpret_cast<int32_t*>(scratch + kNoAllocRowTicketOff);
  a.seq_ticket = reinterpret_cast<int32_t*>(scratch + kNoAllocSeqTicketOff);
  a.splits = splits;
  a.chunk_vec = chunk_vec;
  accept_kernel<<<dim3(splits, rows), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? MARS_OK : MARS_ERR_CUDA;
}
