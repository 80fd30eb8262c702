/*
 * hashevict.h — C ABI of the B300 HashEvict decode-step library (libhashevict.so).
 *
 * The operation ("HashEvict: A Pre-Attention KV Cache Eviction Strategy using
 * Locality-Sensitive Hashing", arXiv 2412.16187; abstract and the technical
 * framework of the method section, steps 1-5):
 *   per decode step and per (batch, KV head),
 *   1-2. project the current query heads and the current key onto a shared
 *        Gaussian matrix W[head_dim][bits] and binarise by sign into `bits`-bit codes;
 *   3.   score every cached key by the Hamming distance between its stored code
 *        and the query codes (summed over the G = heads / kv_heads query heads
 *        of the KV group);
 *   4.   evict the most dissimilar cached token (largest distance; ties go to
 *        the lowest slot) before any attention is computed;
 *   5.   write the current token's key, value and code into the evicted slot;
 *   then attend: out = softmax(q K^T / sqrt(head_dim)) V over the retained
 *   cache (which now holds the current token), as every decode step does
 *   (TTKV page, introduction).
 *   While fewer than `budget` tokens are cached the current token is appended
 *   to the next free slot instead (no scoring).
 *
 * Conventions for every entry point:
 *   - Return 0 (HE_OK) on success, a negative HE_E* code on failure; nothing
 *     aborts.  he_strerror() names a code.  A CUDA error seen by the library is
 *     returned as HE_ECUDA and remembered: the handle then refuses further work.
 *   - Element type: HE_DTYPE_BF16 (bf16 bit patterns, 2 bytes) or HE_DTYPE_FP32.
 *     q, k, v, K, V and W all use the handle's element type.  Outputs are fp32.
 *   - "device" pointers are CUDA device memory of the device current when the
 *     handle was created; "host" pointers are host memory.  Every pointer must
 *     be 16-byte aligned.  Caller-owned buffers stay owned by the caller.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls that
 *     take a stream are asynchronous on it; calls that take host buffers
 *     synchronise the handle's last-used stream first.
 *   - A handle is not thread-safe; use one handle per layer and per thread.
 *   - libhashevict_debug.so exports the same entry points with device-side
 *     bounds checks on every computed global access of the step kernels; a
 *     failed check is returned as HE_EDEVICE by the next synchronising call.
 */
#ifndef HASHEVICT_H
#define HASHEVICT_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HE_OK 0
#define HE_EINVAL (-1)      /* bad configuration, size, pointer or alignment */
#define HE_ENOTFILLED (-2)  /* he_step before he_fill */
#define HE_ECUDA (-3)       /* a CUDA call failed (sticky for the handle) */
#define HE_ENOMEM (-4)      /* device allocation failed */
#define HE_EDEVICE (-5)     /* a kernel reported an internal error (wait gave up) */

#define HE_DTYPE_BF16 0
#define HE_DTYPE_FP32 1

#define HE_VFMT_ELEM 0  /* values stored in the element type */
#define HE_VFMT_INT8 1  /* values stored as int8 rows with one fp32 scale per slot (bf16 only) */
#define HE_VFMT_FP8 2   /* values stored as fp8 E4M3 rows with one fp32 scale per slot (bf16 only) */

/* Handle configuration.  Supported: head_dim in {64, 128};
 * G = heads / kv_heads in {1, 2, 4, 8}; bits in {8, 16, 32, 64};
 * 1 <= budget <= 2^24; batch * kv_heads <= 2^16; dtype HE_DTYPE_*;
 * threshold finite; 0 <= decay <= 1; v_format HE_VFMT_*; 0 <= chunk <= 16
 * (chunk >= 2: bf16, budget % chunk == 0, decay 0, v_format HE_VFMT_ELEM);
 * engine HE_ENGINE_* (HE_ENGINE_FUSED: bf16, decay 0, v_format HE_VFMT_ELEM,
 * chunk <= 1); tau_mode HE_TAU_*.
 * A zero-initialised tail (threshold 0, decay 0, v_format 0, chunk 0, engine 0,
 * tau_mode 0) is the method as the paper describes it.
 * Rows per (batch, KV head): R = budget + chunk - 1 with chunk >= 2, else
 * R = budget; the state calls below return R rows per unit. */
typedef struct {
  int32_t batch;
  int32_t heads;     /* query heads */
  int32_t kv_heads;  /* key/value heads; heads % kv_heads == 0 */
  int32_t head_dim;  /* D */
  int32_t bits;      /* code length b (projection width) */
  int32_t budget;    /* cache slots per (batch, KV head) */
  int32_t dtype;     /* HE_DTYPE_BF16 or HE_DTYPE_FP32 */
  float threshold;   /* binarisation threshold tau: bit j = (projection_j > tau), the
                        "binarisation threshold" design choice of the method section;
                        0 = the sign test */
  uint64_t seed;     /* draws W; one handle (and one seed) per layer */
  float decay;       /* score memory gamma: every resident slot keeps a score
                        A = fmaf(gamma, A, d) (fp32) updated at each evicting step
                        (d its group-summed Hamming distance); the largest A is
                        evicted (ties: lowest slot); a written or filled slot starts
                        at A = 0.  0 = the step's own distances (the paper's method) */
  int32_t v_format;  /* HE_VFMT_ELEM; HE_VFMT_INT8: each value row v is stored as
                        q = v / s rounded half to even with s = max|v| / 127 (fp32), and
                        attended as q * s; HE_VFMT_FP8: stored as c = the E4M3 value
                        (OCP 8-bit floating point format: 4 exponent bits, bias 7,
                        3 mantissa bits, subnormals, largest finite 448) nearest to
                        v / s, ties to the even mantissa, with s = max|v| / 448 (fp32),
                        and attended as c * s.  Keys, codes and evictions are unchanged
                        (the DASH-KV page's value compression; the TTKV page's keys
                        with more bits than values) */
  int32_t chunk;     /* chunk eviction c (the ChunkKV page's chunks of contiguous
                        tokens applied to the method's scores): the budget is cut into
                        budget / c aligned chunks of c slots, a chunk scores the sum of
                        its slots' distances; once the cache is full, new tokens are
                        staged (and attended) in the c - 1 rows after the budget, and
                        the token that would overflow the stage evicts the chunk with
                        the largest score (ties: lowest chunk): the staged tokens in
                        arrival order, then that token, take the chunk's slots.
                        0 or 1 = the method (one slot at a time) */
  int32_t engine;    /* bf16 handles: HE_ENGINE_PIPELINE (0) runs a step as three
                        kernels (attention stream; codes and eviction alongside it;
                        merge and overwrite); HE_ENGINE_FUSED (1) runs it as one
                        kernel (a hash warp per CTA, and the last CTA of each (batch,
                        KV head) merges it; the method only: threshold allowed, no
                        score memory, quantised values or chunks).  Same results. */
  int32_t tau_mode;  /* HE_TAU_FIXED: every bit's threshold is `threshold`;
                        HE_TAU_MEDIAN: one threshold per bit and (batch, KV head),
                        the lower median of the projections of that unit's keys
                        passed to he_fill onto column j of W (element (n - 1) / 2,
                        counting from 0, of the ascending fp32 projections; n = 0
                        gives 0), so that each bit splits the filled keys in half;
                        fixed until the next he_fill.  `threshold` is then unused
                        (the method section's binarisation-threshold design
                        choice, read per bit) */
} he_cfg;

#define HE_TAU_FIXED 0
#define HE_TAU_MEDIAN 1

#define HE_ENGINE_PIPELINE 0
#define HE_ENGINE_FUSED 1

typedef struct he_ctx* he_handle;

/* Creates a handle on the current CUDA device and allocates, in device memory
 * owned by the handle: the cache K, V [batch][kv_heads][R][head_dim], the
 * codes [batch][kv_heads][R] (bits/8-byte words), W [head_dim][bits] drawn
 * from cfg->seed (see he_get_projection) and the step's scratch.
 * Errors: HE_EINVAL (cfg or out NULL, unsupported sizes), HE_ENOMEM, HE_ECUDA. */
int he_create(const he_cfg* cfg, he_handle* out);

/* Fills the cache with n <= budget prompt tokens and codes their keys
 * (method steps 1-2 applied to the cached keys; with tau_mode HE_TAU_MEDIAN it
 * first sets the per-bit thresholds from these keys, using stream-ordered
 * scratch of up to 1 GiB, or one unit's bits * n floats if more).  K, V: device
 * [batch][kv_heads][n][head_dim].  n = 0 empties the cache (K, V may be NULL).
 * Errors: HE_EINVAL (NULL handle, n out of range, NULL or misaligned K/V),
 * HE_ENOMEM (the threshold scratch), HE_ECUDA.  A fill that fails after its
 * checks leaves the handle unfilled: he_step returns HE_ENOTFILLED until a
 * fill succeeds. */
int he_fill(he_handle h, const void* K, const void* V, int32_t n, void* stream);

/* One decode step (method steps 1-5, then attention).  bf16 handles launch
 * three kernels on `stream` (attention partials over the cache, codes and
 * eviction, then merge and overwrite), chained by programmatic dependent
 * launch, or one kernel with HE_ENGINE_FUSED; fp32 handles launch one fused
 * kernel.  The step's kernels may start before the preceding work on `stream`
 * has finished and read q, k, v (and fetch cache tiles) before they wait for
 * it: q, k and v must be complete when he_step is called, or be written by
 * work that does not let dependent launches start early.
 * q: device [batch][heads][head_dim]; k, v: device [batch][kv_heads][head_dim];
 * out: device fp32 [batch][heads][head_dim].  Updates the cache in place.
 * Errors: HE_EINVAL (NULL handle or pointer, misalignment), HE_ENOTFILLED, HE_ECUDA. */
int he_step(he_handle h, const void* q, const void* k, const void* v, float* out, void* stream);

/* he_step on HOST buffers (same shapes): copies q, k, v to handle-owned device
 * staging buffers, runs the step, copies out back and synchronises `stream`.
 * Returns when out is written.  Errors: as he_step. */
int he_step_host(he_handle h, const void* q, const void* k, const void* v, float* out,
                 void* stream);

/* Frees everything the handle owns.  NULL-safe.  Synchronises the device. */
int he_destroy(he_handle h);

/* Slots written by the last step, host [batch][kv_heads]: the evicted slot (with
 * chunk eviction, the evicted chunk's first slot), or -1 when the token was
 * appended to a cache not yet full (or staged).  Synchronises.
 * Also returns HE_EDEVICE if a kernel of this handle reported an internal error. */
int he_last_evicted(he_handle h, int32_t* host_slots);

/* Snapshot of the cache into host buffers (any may be NULL):
 * K, V [batch][kv_heads][R][head_dim] (element type; V bytes with a
 * quantised value cache), codes [batch][kv_heads][R] (bits/8-byte words), occupancy
 * (one int: resident rows, staged ones included).  Synchronises. */
int he_read_state(he_handle h, void* K, void* V, void* codes, int32_t* occupancy);

/* The projection matrix W [head_dim][bits] (element type), host.  W[d][j] is a
 * counter-based N(0,1) draw: st = SplitMix64(seed ^ 0x48455F50524F4A57); for
 * element e = d*bits + j, three SplitMix64(st + 3e + r) give twelve 16-bit
 * integers u; W = (sum u - 393210) / 65536, rounded to bf16 (nearest-even) for
 * bf16 handles.  Synchronises. */
int he_get_projection(he_handle h, void* host_W);

/* Codes of n vectors (method steps 1-2): x device [n][head_dim] (element type),
 * codes device [n] words of bits/8 bytes.  bit j = (sum_d x[d] W[d][j] > threshold),
 * the sum in fp32, fused multiply-add, d = 0..head_dim-1 in order from +0.
 * Errors: HE_EINVAL (also for a handle with tau_mode HE_TAU_MEDIAN, whose
 * thresholds belong to each (batch, KV head)), HE_ECUDA. */
int he_codes(he_handle h, const void* x, int32_t n, void* codes, void* stream);

/* Group-summed Hamming distances of every resident slot to the step's query
 * (method step 3) without changing the cache: q device [batch][heads][head_dim],
 * dist device int32 [batch][kv_heads][R] (slots >= occupancy get 0).
 * Errors: HE_EINVAL, HE_ENOTFILLED, HE_ECUDA. */
int he_scores(he_handle h, const void* q, int32_t* dist, void* stream);

/* Per-slot value scales of a handle with a quantised value cache (v_format
 * HE_VFMT_INT8 or HE_VFMT_FP8), host fp32 [batch][kv_heads][budget]; he_read_state
 * then returns the value rows as bytes [batch][kv_heads][budget][head_dim] (int8
 * values, or E4M3 codes).
 * Synchronises.  Errors: HE_EINVAL (NULL arguments, or another value format). */
int he_read_vscales(he_handle h, float* host_scales);

/* Binarisation thresholds, host fp32 [batch][kv_heads][bits]: the per-bit
 * medians of a handle with tau_mode HE_TAU_MEDIAN (as of its last he_fill), else
 * `threshold` in every entry.  Synchronises (median mode).
 * Errors: HE_EINVAL (NULL arguments), HE_ECUDA, HE_EDEVICE. */
int he_read_thresholds(he_handle h, float* host_tau);

/* Per-slot eviction scores A of a handle with score memory (decay > 0), host
 * fp32 [batch][kv_heads][budget] (slots >= occupancy hold 0).  Synchronises.
 * Errors: HE_EINVAL (NULL arguments, or a handle without score memory). */
int he_read_scores(he_handle h, float* host_scores);

/* Number of resident tokens (host-side state; no synchronisation). */
int he_occupancy(he_handle h, int32_t* occupancy);

/* Algorithmic HBM bytes of one full-cache step (read of retained K, V and codes,
 * write of the overwritten slot, q/k/v in, out, W; with score memory also the
 * read and write of every slot's score) — the roofline numerator. */
int he_step_bytes(he_handle h, uint64_t* bytes);

/* Launch shape of the cache-streaming kernel for the current occupancy: CTAs,
 * CTAs per SM, cache tiles (64 slots each for bf16 handles, 32 for fp32) and
 * pipeline stages. */
int he_launch_info(he_handle h, int32_t* ctas, int32_t* ctas_per_sm, int32_t* tiles,
                   int32_t* stages);

/* Kernel timing mode.  After he_profile_start(h, max_steps) the next max_steps
 * he_step calls record CUDA events on their stream before the cache-streaming
 * kernel and after each of the step's kernels.  The events serialise the
 * kernels (a timed bf16 step does not overlap its codes/eviction kernel with the
 * cache stream, nor the next step with this one), so time steps this way in a
 * pass of their own.  he_profile_stop sums the elapsed times over the recorded
 * steps into ms[4]: [0] the cache-streaming attention kernel (the one fused
 * kernel for fp32 handles), [1] the codes/eviction kernel (0 for fp32), [2] the
 * merge/overwrite kernel (0 for fp32), [3] the whole step; *steps = steps
 * recorded.  It synchronises on the events and leaves timing mode.
 * Errors: HE_EINVAL (NULL handle or pointers, max_steps outside 1..65536),
 * HE_ENOMEM (events could not be created), HE_ECUDA. */
int he_profile_start(he_handle h, int32_t max_steps);
int he_profile_stop(he_handle h, float* ms, int32_t* steps);

/* Number of times, since he_fill, that the attention partial holding the
 * evicted slot was recomputed exactly instead of having the slot's weight
 * subtracted (the slot carried more than half of that partial's softmax mass;
 * with chunk eviction: the chunk outweighed 16 times the weight that remains in
 * the unit).  Always 0 for fp32 handles.  Synchronises. */
int he_recompute_count(he_handle h, int64_t* total);

/* Test export: a per-step eviction log kept on the device.  After
 * he_set_evict_log(h, log, count, capacity), each later step writes, for every
 * unit u = b * kv_heads + j, the slot it wrote (as he_last_evicted reports it)
 * to log[count[u]][u] and then increments count[u]; entries beyond `capacity`
 * are counted but not stored.  log: device int32 [capacity][batch * kv_heads];
 * count: device int32 [batch * kv_heads], set by the caller (normally to 0).
 * The writes happen on the device in step order, so steps issued back to back
 * on a stream, or replayed from a captured CUDA graph, are logged without any
 * host synchronisation; a graph records the log pointers it was captured with.
 * log = NULL turns the log off.  The buffers stay owned by the caller and must
 * outlive every step that logs into them.
 * Errors: HE_EINVAL (NULL handle; log without count or with capacity < 1). */
int he_set_evict_log(he_handle h, int32_t* log, int32_t* count, int32_t capacity);

/* Test export: the distances the step itself computes (method step 3).  After
 * he_set_dist_log(h, dist), each later step that scores a full cache writes the
 * group-summed Hamming distance of every slot it scores to dist[b][j][s]
 * (device int32 [batch][kv_heads][R]); with chunk eviction that is every slot
 * of the budget, the chunks' sums being built from them.  Steps that append
 * write nothing.  NULL turns it off.  Caller-owned, as for the eviction log.
 * Errors: HE_EINVAL (NULL handle). */
int he_set_dist_log(he_handle h, int32_t* dist);

/* Checks of the failure paths.
 * he_set_alloc_limit: a process-wide cap, in bytes, on the device memory one
 * he_create may allocate, and on the scratch of one he_fill with per-bit
 * median thresholds (0 = no cap, the default).  A handle that would need more
 * fails with HE_ENOMEM before allocating anything, and such a fill with
 * HE_ENOMEM (leaving the handle unfilled), as on an exhausted device.  Always
 * returns HE_OK.
 * he_wait_probe: launches on `stream` one kernel that waits on a barrier that
 * nothing completes, through the same bounded wait as every kernel of the
 * library, giving up after limit_us microseconds (1 .. 1,000,000).  On giving
 * up it records the handle's device error flag and exits, as a step kernel
 * does: the next synchronising call on the handle returns HE_EDEVICE and the
 * handle refuses further work; other handles and the CUDA context stay usable.
 * Errors: HE_EINVAL (NULL handle, limit out of range), HE_ECUDA. */
int he_set_alloc_limit(uint64_t bytes);
int he_wait_probe(he_handle h, uint32_t limit_us, void* stream);

/* Allocation-free decode attention.  This entry point has no counterpart in
 * the method's description: it is an integration aid for callers that cannot
 * let a library allocate device memory — runtimes whose device memory is owned
 * by their own pool or arena (a second allocator would fragment it or break
 * its accounting), deployments that fix every byte of device memory up front.
 *   out[b][h][:] = sum_{s < n} softmax_s(q[b][h] . K[b][kv][s] / sqrt(head_dim))
 *                  V[b][kv][s],   kv = h / (heads / kv_heads)
 * K, V: device bf16 [batch][kv_heads][budget][head_dim] (rows s >= n of each
 * (batch, kv) are read and ignored: they must hold finite values); q: device
 * bf16 [batch][heads][head_dim]; out: device fp32 [batch][heads][head_dim].
 * The same split-K tensor-core kernel as he_step runs with its partial results
 * in one static device array of HE_NOALLOC_SCRATCH_BYTES per GPU (every GPU that
 * loads the library holds it until the process exits).  Limit: with C = min(the
 * number of 64-slot tiles, SMs x resident CTAs per SM) and R = 4 * (4 *
 * ceil(2G / 4) + G * head_dim) bytes per partial record (G = heads / kv_heads),
 * (C + batch * kv_heads) * R + 256 <= HE_NOALLOC_SCRATCH_BYTES, else HE_EINVAL.
 * The first call on each device does a one-off set-up (the array's device
 * address, kernel attributes) on the current device.  Not thread-safe on a
 * device's first call.  Every
 * call uses the same array, so calls that overlap on the GPU race: order them
 * (one stream, or events).  Each call clears the array's error word itself
 * (an asynchronous memset on `stream`); nothing else in the array needs to
 * start at zero.  No cudaMalloc or cudaFree is called.
 * Device-side failure: if a kernel of the call gives up a bounded wait, the
 * call's whole output is NaN (the call has already returned HE_OK by then).
 * Errors: HE_EINVAL (sizes, NULL or misaligned pointers, scratch too small),
 * HE_ECUDA. */
#define HE_NOALLOC_SCRATCH_BYTES (8u << 20)
int he_attend_noalloc(int32_t batch, int32_t heads, int32_t kv_heads, int32_t head_dim,
                      int32_t budget, int32_t n, const void* K, const void* V, const void* q,
                      float* out, void* stream);

/* Human-readable name of a return code. */
const char* he_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* HASHEVICT_H */
