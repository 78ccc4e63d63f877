/*
 * mars.h - C ABI of libmars, the GB300 (sm_103a) hot path of MARS
 * (Mask AutoRegreSsion) multi-token generation.
 *
 * Method sources, cited by page title and section / equation:
 *   [paper] "MARS: Enabling Autoregressive Models Multi-Token Generation"
 *           (arXiv 2604.07023).
 *   [blog]  the authors' MARS blog post (xalp.net/posts/2026-06-mars).
 *   [news]  "MARS: 자기회귀 모델의 멀티 토큰 생성을 가능하게 하는 기법" (aitrends.kr).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Tensors are caller-owned DEVICE pointers, dense row-major in the shapes
 *   written beside each argument.  bf16 values are passed as their 16-bit
 *   patterns (uint16_t), i.e. the storage of __nv_bfloat16 / torch.bfloat16.
 * - Alignment: bf16 tensors must be 16-byte aligned (they are moved with 16-byte
 *   vector, cp.async and TMA accesses), except `logits`, which needs only 2-byte
 *   alignment; int32 / fp32 arrays need 4-byte alignment.
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *   stream) and never allocate, free or synchronise.  The calls other than
 *   mars_accept_noalloc can be captured in a CUDA graph.
 * - Kernels are launched as programmatic dependent launches: their set-up may
 *   overlap the tail of the previous kernel in the stream, but none of them
 *   touches global memory before that kernel has completed, so stream order
 *   holds as for plain launches.
 * - The return value reports what the host can see before launch; conditions
 *   that only the device can see are OR-ed into the optional device status
 *   word (`int32_t*` in device memory, may be NULL), which the caller reads
 *   after the stream has completed and clears when it wants to.
 * - Inputs must be finite.  The result for NaN / Inf inputs is unspecified
 *   (no fault: it is only arithmetic on the values).
 * - GQA: query head h reads KV head h / (Hq / Hkv) (contiguous groups).
 */
#ifndef MARS_H_
#define MARS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Host-visible return codes. */
#define MARS_OK 0
#define MARS_ERR_INVALID_ARG 1         /* null / misaligned pointer, bad size, unsupported shape */
#define MARS_ERR_WORKSPACE_TOO_SMALL 2 /* workspace smaller than the *_workspace_size() answer */
#define MARS_ERR_CUDA 3                /* a CUDA runtime call or a launch failed */
#define MARS_ERR_UNSUPPORTED_DEVICE 4  /* current device is not compute capability 10.3 */
#define MARS_ERR_SCRATCH_LIMIT 5       /* shape too large for mars_accept_noalloc's fixed scratch */
#define MARS_ERR_SCRATCH_NOT_READY 6   /* mars_accept_noalloc's first call in a CUDA context came during a stream
                                          capture; make one call outside capture first */

/* Bits that kernels OR into the device status word. */
#define MARS_DEV_CAPACITY 1   /* mars_accept: cache_len + n_commit would exceed cap; that sequence was not appended;
                                 mars_decode_attn_deferred: cache_len + pending > cap; that sequence's output is zero */
#define MARS_DEV_LEN_RANGE 2  /* mars_decode_attn: a cache_len[b] was < 0 or > max_len; that sequence's output is zero */
#define MARS_DEV_TIMEOUT 4    /* mars_train_attn(_bwd), mars_decode_attn, mars_accept: an internal pipeline wait hit
                                 its iteration limit; output incomplete */

/* Human-readable text for a return code (static storage, never NULL). */
const char* mars_status_string(int status);

/* Text of the CUDA error behind the calling thread's last MARS_ERR_CUDA
 * ("no error" if there was none); static storage, never NULL. */
const char* mars_last_cuda_error(void);

/* Library ABI version: 100 * major + minor. */
int mars_version(void);

/*
 * mars_train_attn - attention over the concatenated sequence z = [x ; x~]
 * under the MARS structured mask ([paper] Sec. 3.2, Eq. 1 and Eq. 2).
 *
 * Positions 0..L-1 of z are the clean stream, L..2L-1 the noisy ([MASK])
 * stream.  With 0-indexed query i and key j:
 *   clean query (i < L):       sees clean keys j <= i                    (causal)
 *   noisy query i = L + t:     sees clean keys j < B * floor(t / B)       (earlier blocks)
 *                              and noisy keys L + u with floor(u / B) == floor(t / B), u <= t
 * L need not be a multiple of B (the last block is short).
 *
 *   q    [batch, 2L, Hq,  D]  bf16          o   [batch, 2L, Hq, D] bf16 (written)
 *   k, v [batch, 2L, Hkv, D]  bf16          lse [batch, Hq, 2L] fp32, natural-log
 *                                               log-sum-exp of the scaled masked
 *                                               scores (may be NULL)
 *   scale: multiplies q.k (normally 1/sqrt(D)).
 * Supported: D in {64, 128}; Hq % Hkv == 0; 1 <= B; 1 <= L <= 65536.
 * Fully masked tiles are skipped; no workspace.
 */
int mars_train_attn(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                    uint16_t* o, float* lse,
                    int batch, int L, int B, int Hq, int Hkv, int D, float scale,
                    int32_t* status, void* stream);

/*
 * mars_train_attn_bwd - gradients of mars_train_attn with respect to q, k and
 * v ([paper] Sec. 3.2: both streams share one forward, so one backward carries
 * the gradients of the training losses, Eqs. 3 and 5, to q, k and v).
 *
 * For every head, with S = scale q k^T, P = softmax(S + M) (the Eq. 2 mask,
 * recomputed from the forward's log-sum-exp: P = exp(S - lse)) and dO the
 * gradient of o:
 *   dV = P^T dO,  dP = dO v^T,  dS = P * (dP - rowsum(dO * o)),
 *   dQ = scale dS k,  dK = scale dS^T q,
 * and with GQA every query head of a group adds its dK, dV to the group's KV
 * head.  P and dS are rounded to bf16 for the tensor-core products, every
 * accumulation is fp32, the outputs are bf16.
 *
 *   q, o, dout [batch, 2L, Hq, D] bf16        dq [batch, 2L, Hq, D] bf16 (written)
 *   k, v       [batch, 2L, Hkv, D] bf16       dk, dv [batch, 2L, Hkv, D] bf16 (written)
 *   lse        [batch, Hq, 2L] fp32 (the forward's, natural log)
 *   workspace  device buffer of >= mars_train_attn_bwd_workspace_size(batch,
 *              L, Hq, Hkv, D) bytes (it holds rowsum(dO * o), two work counters
 *              and, when Hq > Hkv, fp32 dK, dV partials of the GQA groups that
 *              are split into chunks of query heads); contents on entry do not
 *              matter; calls that share it must not overlap in time.
 * Kernel launches on `stream`: the row sums; dK and dV per (KV head, key tile,
 * chunk of the group's query heads); the sum of the chunks where a group was
 * split (when Hq > Hkv); then dQ per (query head, query tile).
 * Persistent CTAs take work units from an atomic counter, but every output
 * element comes from one fixed sequence of operations whichever CTA runs it, so
 * the result is deterministic.  Supported: D in {64, 128}; Hq % Hkv == 0; 1 <= B;
 * 1 <= L <= 65536.  All pointers 16-byte aligned except lse (4 bytes).
 */
size_t mars_train_attn_bwd_workspace_size(int batch, int L, int Hq, int Hkv, int D);
int mars_train_attn_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const uint16_t* o, const uint16_t* dout, const float* lse,
                        uint16_t* dq, uint16_t* dk, uint16_t* dv,
                        int batch, int L, int B, int Hq, int Hkv, int D, float scale,
                        void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/*
 * mars_decode_attn - attention of one sliding-window decode step
 * ([paper] Fig. 2 right: B [MASK] tokens appended after the cursor and
 * filled by one forward; [blog] "Inference: a knob, not a mode switch").
 *
 * Query i (0 <= i < B) of sequence b sees the cache_len[b] committed keys of
 * its KV head and the new keys c <= i of this step (causal among the
 * placeholders, as in the noisy intra-block case of Eq. 2).
 *
 *   q              [batch, B, Hq, D]     bf16
 *   k_new, v_new   [batch, B, Hkv, D]    bf16  (K/V of this step's B positions)
 *   k_cache, v_cache [batch, Hkv, cap, D] bf16 (block-level KV cache, read only)
 *   cache_len      [batch] int32, device; every value in [0, max_len]
 *   o              [batch, B, Hq, D]     bf16 (written)
 * Supported: D in {64, 128}; 1 <= B <= 16; Hq % Hkv == 0; max_len <= cap.
 * A cache_len outside [0, max_len] sets MARS_DEV_LEN_RANGE and that
 * sequence's output is written as zeros.  No workspace.
 */
/*
 * mars_decode_attn_workspace_size - bytes of workspace mars_decode_attn needs,
 * which is always 0 (it takes none).  The splits of one unit's cache are merged
 * inside its thread-block cluster through distributed shared memory, so no
 * partial result goes through global memory.  The query exists for callers
 * written against a split-K decode call that asks for its workspace first.
 */
size_t mars_decode_attn_workspace_size(int batch, int B, int Hq, int D, int max_len);
int mars_decode_attn(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                     const uint16_t* k_cache, const uint16_t* v_cache,
                     const int32_t* cache_len,
                     int batch, int B, int Hq, int Hkv, int D, int cap, int max_len,
                     float scale, uint16_t* o, int32_t* status, void* stream);

/*
 * mars_decode_attn_deferred - the decode step of the deferred-KV sampler (the
 * authors' MARS blog post, "Inference: a knob, not a mode switch": KV
 * commitment is deferred into the next proposal forward, with per-sample
 * cursors and a cache-validity bitmask, so that no extra forward, cache copy
 * or batch-wide barrier commits the accepted tokens).
 *
 * The forward of this step carries S = 2B slots per sequence.  Slots 0..B-1
 * hold the tokens that the previous step committed, fed back as ordinary
 * tokens; slot c is valid while c < pending[b] (the previous step's n_commit).
 * Slots B..2B-1 hold the B new [MASK] placeholders and are always valid.  The
 * valid slots follow the cache_len[b] committed cache rows in slot order:
 * a valid query slot sees every committed cache row and the valid slots up to
 * and including itself (causal, as in the noisy intra-block case of Eq. 2).
 * The output row of an invalid slot is zero, and nothing an invalid slot holds
 * (even NaN) reaches a valid row.  The K/V rows of the valid pending slots are
 * written into the cache at rows cache_len[b] .. cache_len[b] + pending[b] - 1;
 * cache_len itself is advanced by mars_accept_ex with MARS_ACCEPT_DEFERRED.
 *
 *   q              [batch, 2B, Hq, D]     bf16
 *   k_new, v_new   [batch, 2B, Hkv, D]    bf16  (K/V of this step's 2B slots)
 *   k_cache, v_cache [batch, Hkv, cap, D] bf16  (read; the pending rows written)
 *   cache_len      [batch] int32, device; every value in [0, max_len]
 *   pending        [batch] int32, device; every value in [0, B]
 *   o              [batch, 2B, Hq, D]     bf16 (written)
 * Supported: D in {64, 128}; 1 <= B <= 8; Hq % Hkv == 0; max_len <= cap.
 * A cache_len outside [0, max_len] or a pending outside [0, B] sets
 * MARS_DEV_LEN_RANGE, and cache_len + pending > cap sets MARS_DEV_CAPACITY;
 * either way that sequence's output is written as zeros and its cache is not
 * written.  Other CTAs of the same sequence may read the rows being written
 * inside their last cache tile; those rows are masked.  No workspace.
 */
int mars_decode_attn_deferred(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                              uint16_t* k_cache, uint16_t* v_cache,
                              const int32_t* cache_len, const int32_t* pending,
                              int batch, int B, int Hq, int Hkv, int D, int cap, int max_len,
                              float scale, uint16_t* o, int32_t* status, void* stream);

/*
 * mars_accept - confidence-threshold acceptance with the block-level KV
 * append ([blog] "Inference: a knob, not a mode switch": commit left to right
 * while the top-1 probability holds, stop at the first position below tau;
 * [paper] Sec. 3.1 gap (4): strictly left-to-right; [news]: at least one
 * token is always accepted; [paper] contributions: block-level KV cache).
 *
 * For each row (b, i):  m = max_v logits, tokens = smallest v with logits == m,
 *                       conf = 1 / sum_v exp(logits - m)   (top-1 probability)
 * For each sequence b:  n = number of leading i with conf >= tau, then max(n, 1);
 *                       rows 0..n-1 of k_new / v_new are copied to cache
 *                       positions cache_len[b] .. cache_len[b]+n-1 and
 *                       cache_len[b] += n.
 *
 *   logits           [batch, B, V] bf16
 *   k_new, v_new     [batch, B, Hkv, D] bf16
 *   k_cache, v_cache [batch, Hkv, cap, D] bf16 (updated in place)
 *   cache_len        [batch] int32, device, in/out
 *   tokens [batch, B] int32, conf [batch, B] fp32, n_commit [batch] int32 (written)
 *   workspace        device buffer of >= mars_accept_workspace_size(batch, B, V)
 *                    bytes, ZERO-FILLED BEFORE ITS FIRST USE (cudaMemset,
 *                    torch.zeros).  It holds one partial result per slice of
 *                    logits (4 to 16 KB), one count per sequence (batch-minimum
 *                    mode of mars_accept_ex) and one ticket per sequence; every
 *                    call leaves the tickets at zero again, so a workspace is
 *                    zeroed once and then reused.  Calls that share a workspace
 *                    must not overlap in time.
 * The call is one kernel launch on `stream`: persistent CTAs stream the logits
 * in slices; the warp that reduces the last slice of a sequence (an atomic
 * ticket per sequence, no waiting) applies the commit rule and appends.
 * (The batch-minimum mode of mars_accept_ex adds two short launches.)
 * If cache_len[b] + n > cap nothing is appended for b, cache_len[b] is kept,
 * n_commit[b] is 0 and MARS_DEV_CAPACITY is set.
 * Supported: 1 <= B <= 16, 1 <= V, D % 8 == 0, D <= 256.
 */
size_t mars_accept_workspace_size(int batch, int B, int V);
int mars_accept(const uint16_t* logits, int batch, int B, int V, float tau,
                const uint16_t* k_new, const uint16_t* v_new,
                uint16_t* k_cache, uint16_t* v_cache, int32_t* cache_len,
                int Hkv, int D, int cap,
                int32_t* tokens, float* conf, int32_t* n_commit,
                int32_t* status, void* workspace, size_t workspace_bytes, void* stream);

/*
 * mars_accept_ex - mars_accept with options, `flags` an OR of:
 *   MARS_ACCEPT_MARGIN     conf is the margin p1 - p2 (see mars_accept_margin);
 *   MARS_ACCEPT_BATCH_MIN  every sequence commits n = min over the batch of the
 *                          per-sequence counts (each at least one) and appends n
 *                          rows: the paper's original sampler, whose block-level
 *                          cache moved forward by the smallest acceptance in the
 *                          batch (the authors' MARS blog post, "Inference: a knob,
 *                          not a mode switch").  n_commit[b] = n for every b; one more launch
 *                          (one CTA per sequence) takes the minimum and appends.
 *                          A sequence for which cache_len[b] + n > cap sets
 *                          MARS_DEV_CAPACITY, commits 0 and is left unchanged.
 *   MARS_ACCEPT_DEFERRED   the acceptance step of the deferred-KV sampler (see
 *                          mars_decode_attn_deferred): on entry n_commit[b] holds
 *                          the previous step's count, whose rows this step's
 *                          decode attention has written at the cursor; the call
 *                          sets cache_len[b] += that count, then n_commit[b] =
 *                          this step's count (the next step's pending).  No K/V
 *                          is copied: k_new, v_new, k_cache, v_cache, Hkv and D
 *                          are not read and may be NULL / 0.  Tokens and conf
 *                          are those of the other modes.  If the old count is
 *                          outside [0, B] or cache_len + count > cap, the call
 *                          sets MARS_DEV_CAPACITY, keeps cache_len and commits 0;
 *                          if the new count would not fit after the cursor
 *                          (cache_len + count > cap) it commits 0 and sets
 *                          MARS_DEV_CAPACITY.  Combines with the other flags.
 * Other bits return MARS_ERR_INVALID_ARG.  Arguments, workspace (its size from
 * mars_accept_workspace_size covers both modes) and outputs are those of
 * mars_accept.  mars_accept(...) == mars_accept_ex(..., flags = 0, ...).
 */
#define MARS_ACCEPT_MARGIN 1
#define MARS_ACCEPT_BATCH_MIN 2
#define MARS_ACCEPT_DEFERRED 4
int mars_accept_ex(const uint16_t* logits, int batch, int B, int V, float tau, int flags,
                   const uint16_t* k_new, const uint16_t* v_new,
                   uint16_t* k_cache, uint16_t* v_cache, int32_t* cache_len,
                   int Hkv, int D, int cap,
                   int32_t* tokens, float* conf, int32_t* n_commit,
                   int32_t* status, void* workspace, size_t workspace_bytes, void* stream);

/*
 * mars_accept_margin - mars_accept with the margin gate.  The authors' MARS blog
 * post ("Inference: a knob, not a mode switch") reports that a gate on the top
 * token's lead over the rest, instead of on its probability, does better on
 * text with strict formatting.  The margin is read as p1 - p2: the top-1 probability
 * minus the largest probability of any other token, at temperature 1.
 *
 * Same arguments, workspace, outputs and error behaviour as mars_accept,
 * except that conf[b, i] holds the margin p1 - p2 (0 when two tokens tie at the
 * maximum, p1 when V == 1) and a position passes while conf >= tau.  It is
 * computed in the same single pass over the logits (the second largest logit
 * is tracked beside the maximum): p1 - p2 = (1 - exp(l2 - m)) / sum exp(l - m).
 */
int mars_accept_margin(const uint16_t* logits, int batch, int B, int V, float tau,
                       const uint16_t* k_new, const uint16_t* v_new,
                       uint16_t* k_cache, uint16_t* v_cache, int32_t* cache_len,
                       int Hkv, int D, int cap,
                       int32_t* tokens, float* conf, int32_t* n_commit,
                       int32_t* status, void* workspace, size_t workspace_bytes, void* stream);

/*
 * mars_lm_head_accept - the LM head of the proposal positions fused with
 * mars_accept.  The authors' MARS blog post ("Where it stands against the
 * alternatives") names the 152k-vocabulary projection that every proposal ends
 * in as the drafter's cost; here its logits
 *     logits[b, i, v] = sum_k hidden[b, i, k] * weight[v, k]
 * are accumulated in fp32 in tensor memory and reduced on the spot to each
 * row's maximum, lowest argmax and sum of exp(logit - max): they are never
 * written to memory.  Tokens, conf (top-1 probability, computed from the fp32
 * logits), the commit rule and the block-level KV append are those of
 * mars_accept.
 *
 *   hidden           [batch, B, K] bf16, the final hidden states of the B proposal
 *                    positions; K a multiple of 64
 *   weight           [V, K] bf16, the head's linear map (one row per vocabulary entry)
 *   workspace        device buffer of >= mars_lm_head_accept_workspace_size(batch,
 *                    B, V) bytes (one partial per row and vocabulary range);
 *                    contents on entry do not matter; calls that share it must
 *                    not overlap in time
 * Other arguments, outputs and error behaviour as mars_accept; hidden and weight
 * must be 16-byte aligned.  Two kernel launches on `stream` (the fused head,
 * then one CTA per sequence for the commit rule and the append).
 */
size_t mars_lm_head_accept_workspace_size(int batch, int B, int V);
int mars_lm_head_accept(const uint16_t* hidden, const uint16_t* weight, int batch, int B, int K, int V, float tau,
                        const uint16_t* k_new, const uint16_t* v_new,
                        uint16_t* k_cache, uint16_t* v_cache, int32_t* cache_len,
                        int Hkv, int D, int cap,
                        int32_t* tokens, float* conf, int32_t* n_commit,
                        int32_t* status, void* workspace, size_t workspace_bytes, void* stream);

/*
 * mars_accept_noalloc - mars_accept for callers that cannot allocate device
 * memory.  The MARS pages have no counterpart to this call: it exists for
 * callers such as plugins that only receive the input and output buffers of a
 * host framework, or serving loops under a fixed memory budget, for which a
 * cudaMalloc could fail mid-decode and would synchronise the device.
 *
 * Same arguments and results as mars_accept, without the workspace.  The
 * scratch is a 1 MiB array inside the library (a file-scope __device__
 * array), which every GPU that loads the library holds until the process
 * exits.  Nothing is allocated or freed by this call; nothing in the array
 * needs to start at zero.
 *   - Limit: batch * B * ceil(V / 8192) <= 65536 (one partial result per
 *     16 KB slice of logits must fit); larger shapes return
 *     MARS_ERR_SCRATCH_LIMIT without launching anything.
 *   - The first call in each CUDA context (per device; again after a
 *     cudaDeviceReset) sets the scratch up: it looks up the array's device
 *     address with that device current.  Make that first call before any
 *     stream capture begins: a first call on a stream that is being captured
 *     returns MARS_ERR_SCRATCH_NOT_READY and launches nothing.
 *   - All calls in the process share the one array per device and it keeps
 *     the last call's contents; calls that overlap on the GPU (for example on
 *     two streams at once) race on it and must be serialised by the caller.
 */
int mars_accept_noalloc(const uint16_t* logits, int batch, int B, int V, float tau,
                        const uint16_t* k_new, const uint16_t* v_new,
                        uint16_t* k_cache, uint16_t* v_cache, int32_t* cache_len,
                        int Hkv, int D, int cap,
                        int32_t* tokens, float* conf, int32_t* n_commit,
                        int32_t* status, void* stream);

/*
 * mars_selftest_wait_timeout - runs, on the device, the bounded pipeline wait
 * that every kernel of this library uses, on a barrier that needs two arrivals.
 * The MARS pages have no counterpart: this checks the library's own failure
 * path without faulting, trapping or hanging the GPU.
 *
 *   withhold_arrival  nonzero: the second arrival never comes, so the wait
 *                     gives up after spin_limit polls; nothing asynchronous
 *                     (no copy, no tensor-core commit) targets the barrier
 *   spin_limit        polls before the wait gives up, 1 .. 2^20 (the kernels'
 *                     own limit, about 4 s on GB300, is the maximum)
 *   status           device int32 word: MARS_DEV_TIMEOUT is OR-ed in when the
 *                     wait gave up (required)
 *   elapsed_ns       device uint64 (8-byte aligned, may be NULL): nanoseconds
 *                     the wait took (%globaltimer)
 * The kernel holds tensor memory across the wait and frees it afterwards, as
 * the real kernels do when a wait gives up, so the context stays usable.
 */
int mars_selftest_wait_timeout(int withhold_arrival, unsigned int spin_limit, int32_t* status,
                               unsigned long long* elapsed_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MARS_H_ */
