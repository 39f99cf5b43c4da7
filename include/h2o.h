/*
 * h2o.h - C ABI of the GB300 (sm_103a) H2O heavy-hitter KV-cache library.
 *
 * H2O keeps, per (batch, head) pair, a fixed budget of C = heavy + recent
 * cached tokens: the `recent` most recent ones plus the `heavy` tokens with the
 * largest accumulated attention score ("H2O: Heavy-Hitter Oracle ... 深度解读报告",
 * sections 3.1, 3.3 and 3.4; "H2O" inference-research notes, summary).
 *
 * Conventions shared by every call
 *  - All tensor arguments are DEVICE pointers owned by the caller, borrowed
 *    for the stream-ordered duration of the call, densely packed, row-major.
 *    B = batch, H = heads, D = head_dim, L = prompt length, P = B*H pairs.
 *  - q / k / v arguments have the cache's K/V dtype (h2o_dtype); outputs are
 *    float32.  Device pointers must be 16-byte aligned.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and never synchronise the host, except the calls marked
 *    "synchronous".  One cache must not be used from two streams at once.
 *  - Return values are h2o_status codes; no exception crosses the ABI.
 *    Argument errors are detected on the host before any launch.  Device-side
 *    checks latch a flag that h2o_cache_check() reports as H2O_EDEVICE.
 *  - h2o_last_error() returns a thread-local message for the last failure.
 *  - The library owns the slot store (K, V), the float32 score buffer, the
 *    int32 position tags, the recent ring and the per-pair counters; they are
 *    allocated in h2o_cache_create and freed in h2o_cache_destroy.
 */
#ifndef H2O_GB300_H
#define H2O_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define H2O_API __attribute__((visibility("default")))
#else
#define H2O_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { H2O_F16 = 0, H2O_F32 = 1 } h2o_dtype;

typedef enum {
  H2O_OK = 0,
  H2O_EINVAL = -1,  /* bad argument (NULL pointer, size out of range, ...) */
  H2O_ENOMEM = -2,  /* device allocation failed */
  H2O_ECUDA = -3,   /* a CUDA runtime call failed (message has the CUDA error) */
  H2O_ESTATE = -4,  /* call not valid in the cache's state (e.g. positions exhausted) */
  H2O_EDEVICE = -5  /* a device-side check fired (see h2o_cache_check) */
} h2o_status;

typedef struct h2o_cache h2o_cache; /* opaque */

/* Preallocate a cache for B x H pairs of `heavy_budget + recent_budget` slots
 * ("... 深度解读报告", section 3.4: preallocated memory, overwrite in place,
 * heavy-hitter region + recent region).  head_dim in {64, 128};
 * heavy_budget >= 0; recent_budget >= 1 (the newest token is always recent);
 * slots <= 65536.  kv_dtype is an h2o_dtype.  The cache starts empty (as after
 * h2o_cache_reset).  Uses the current CUDA device.  *out = NULL on failure. */
H2O_API int h2o_cache_create(int batch, int heads, int head_dim, int heavy_budget, int recent_budget,
                     int kv_dtype, h2o_cache** out);

/* Free every allocation of the cache.  NULL-safe.  The caller must ensure no
 * call on the cache is still running on a stream. */
H2O_API void h2o_cache_destroy(h2o_cache* cache);

/* Prefill ("... 深度解读报告", section 3.4, prefill rule; section 3.3 for the
 * score): for each pair, full causal attention over the prompt,
 * column sums colsum_j = sum_{i>=j} softmax_i(scale * q_i . k_j), then
 *   L <= C : keep every position (slot j = position j);
 *   L >  C : keep positions L-R..L-1 (recent) and the `heavy` positions below
 *            L-R with the largest (colsum, position) keys.
 * Heavy hitters go to slots 0..heavy-1 in ascending position, the recent window
 * to slots heavy..C-1; each kept slot's score = its colsum.  Replaces whatever
 * the cache held.  q, k, v: [B, H, L, D] kv_dtype.  out_or_null: [B, H, L, D]
 * float32 causal attention output, or NULL to skip it.  prompt_len = 0 empties
 * the cache.  The first prefill at a new maximum prompt length allocates its
 * workspaces (cudaMalloc: row statistics and column sums, and with fp16 K/V
 * and an output also the output pass's column-sum partials, 2 KB per pair per
 * pair of 128-token blocks); later ones allocate nothing. */
H2O_API int h2o_prefill(h2o_cache* cache, const void* q, const void* k, const void* v, int prompt_len,
                float scale, float* out_or_null, void* stream);

/* h2o_prefill plus optional float32 views of its intermediate results:
 * colsum_or_null [B, H, L] (every position's column sum) and
 * lse_or_null [B, H, L] (log-sum-exp of each causal row, natural log, of the
 * scaled logits). */
H2O_API int h2o_prefill_ex(h2o_cache* cache, const void* q, const void* k, const void* v, int prompt_len,
                   float scale, float* out_or_null, float* colsum_or_null, float* lse_or_null,
                   void* stream);

/* Ragged batch: h2o_prefill_ex where batch row b's prompt has lengths[b]
 * tokens (clamped to 0..max_len).  The prefill rule ("H2O ... 深度解读报告"
 * §3.4) is applied to every (b, h) pair with its own length: keep all when
 * lengths[b] <= heavy + recent, else the top-heavy column sums of positions
 * < lengths[b] - recent plus the last `recent`; the pair's next decode
 * position is lengths[b] (0: the pair starts empty).  lengths: [B] int32
 * device pointer (4-byte aligned), read on the stream, so it may be written
 * by earlier work on it.  q, k, v: [B, H, max_len, D] with row b valid in
 * positions < lengths[b]; padded positions are read but contribute nothing
 * and must hold finite values (zeros suit).  out_or_null, colsum_or_null,
 * lse_or_null as in h2o_prefill_ex, [B, H, max_len, ...]; their entries at
 * padded positions are unspecified.  max_len = 0 empties the cache.  Not in
 * the pages, which pad every prompt to one length: this serves batches of
 * prompts of different lengths without padding them into the keep rule. */
H2O_API int h2o_prefill_ragged(h2o_cache* cache, const void* q, const void* k, const void* v, int max_len,
                               const int32_t* lengths, float scale, float* out_or_null, float* colsum_or_null,
                               float* lse_or_null, void* stream);

/* One decode step for every pair ("... 深度解读报告", sections 3.1, 3.3, 3.4):
 *   1. attend over the kept slots and the new token: softmax of
 *      scale * q . k over kept + self only; out = sum_j p_j v_j;
 *   2. score[j] += p_j for every kept slot;
 *   3. if the cache is full, evict the kept slot with the lowest
 *      (score, position) among positions <= p - recent; otherwise use the next
 *      free slot;
 *   4. overwrite that slot with k_new / v_new, score = p_self, position = p,
 *      and append it to the recent ring.
 * q, k_new, v_new: [B, H, D] kv_dtype.  out: [B, H, D] float32 (required).
 * evicted_or_null: [B, H] int32, the slot freed this step or -1 while filling.
 * Counters live on the device, so steps can be captured in a CUDA graph and
 * replayed.  Returns H2O_ESTATE when the int32 position would overflow. */
H2O_API int h2o_decode_step(h2o_cache* cache, const void* q, const void* k_new, const void* v_new,
                    float scale, float* out, int32_t* evicted_or_null, void* stream);

/* Empty the cache (count 0, position 0): a stream that starts without a
 * prompt.  Asynchronous on `stream`. */
H2O_API int h2o_cache_reset(h2o_cache* cache, void* stream);

/* Size in bytes of the host image used by export/import. */
H2O_API size_t h2o_cache_state_bytes(const h2o_cache* cache);

/* Synchronous.  Copy the whole cache state into host memory `host_buf` of
 * `bytes` >= h2o_cache_state_bytes().  Layout (little-endian, packed):
 *   int32 header[16] = {magic 0x48324F31, version 1, B, H, D, heavy, recent,
 *                       kv_dtype, 0...}
 *   K      [P, C, D] kv_dtype     V [P, C, D] kv_dtype
 *   score  [P, C]   float32       pos [P, C] int32 (-1 = empty slot)
 *   ring   [P, R]   int32 (-1 = empty)
 *   ctr    [P, 4]   int32 {next position p, count, ring head, 0} */
H2O_API int h2o_cache_export_state(const h2o_cache* cache, void* host_buf, size_t bytes, void* stream);

/* Synchronous.  Load a host image written by export (or built by a caller in
 * the same layout).  The header must match the cache's shape and dtype. */
H2O_API int h2o_cache_import_state(h2o_cache* cache, const void* host_buf, size_t bytes, void* stream);

/* Synchronous.  Wait for the stream, then report H2O_EDEVICE if a device-side
 * check has fired since the last h2o_cache_check (and clear it), or the
 * pending CUDA error as H2O_ECUDA. */
H2O_API int h2o_cache_check(h2o_cache* cache, void* stream);

/* Tuning of the decode kernel's launch shape: `splits` CTAs (one thread-block
 * cluster) share a pair, each streaming its slots through a ring of `stages`
 * 16-row shared-memory stages; splits must be 1, 2, 4, 8 or 16, and stages a
 * multiple of the kernel's consumer warps up to 18: 6, 12 or 18 for one CTA
 * per pair (six consumer warps), 4, 8, 12 or 16 for clusters (four), and 8
 * or 16 for either while position rolling is on (eight).  Or splits =
 * H2O_DECODE_WARP_PER_PAIR: one warp streams a whole pair through its own
 * ring of `stages` (2..8) and then takes its next pair, for many pairs of at
 * most 1024 slots.  0 = automatic for either value (the automatic choice
 * takes warp per pair when there are at least four pairs per SM).  Returns
 * H2O_EINVAL for other values or if the shape cannot be scheduled on the
 * current device.  Every shape computes the same step. */
#define H2O_DECODE_WARP_PER_PAIR (-1)
H2O_API int h2o_cache_set_decode_shape(h2o_cache* cache, int splits, int stages);

/* Position rolling for long or endless streams ("... 深度解读报告", section
 * 4.4: H2O with position rolling on 4-million-token streams).  With
 * rope_base > 0 every decode step takes its logits between rotary-embedded
 * vectors (RoFormer: element pair (2i, 2i+1) rotated by position *
 * rope_base^(-2i/D)) whose positions count inside the cache: the kept tokens
 * are numbered 0..n-1 in text order and the new token gets n.  q, k_new and
 * the cached keys are given, and kept, unrotated.  rope_base = 0 turns it
 * off.  Synchronous: waits for the device and reads the positions back to
 * rank the kept tokens.  While it is on, h2o_prefill, h2o_prefill_ex and
 * h2o_prefill_ragged return H2O_ESTATE (they apply no rotary embedding;
 * decode from an empty or reset cache), and decode runs on the cluster
 * kernel (a warp-per-pair shape is refused; turning it on or off resets the
 * shape to automatic).  Returns H2O_EINVAL for a negative or non-finite base. */
H2O_API int h2o_cache_set_position_rolling(h2o_cache* cache, float rope_base);

/* Tuning of position rolling (no counterpart in the pages; the result of a
 * decode step does not depend on it).  A kept token's rank r is rotated as
 * a product of per-digit rotations: the lowest digit of `low_bits` bits is
 * folded into the query once per step, and each higher digit of `hi_bits`
 * bits costs every key one rotation; the tables take 2^low_bits entries,
 * 2^hi_bits per middle level and what the top digit reaches, each D/2 cos,
 * sin pairs of shared memory per CTA.  Both in 4..6, or both 0 for the
 * automatic choice (the fewest levels whose tables keep the automatic
 * launch shape as resident as the smallest tables would; rolling starts
 * with it).  Synchronous, like h2o_cache_set_position_rolling, and resets
 * the launch shape to automatic.  Returns H2O_ESTATE when rolling is off,
 * H2O_EINVAL for other widths or for widths whose tables cannot be
 * scheduled. */
H2O_API int h2o_cache_set_rolling_digits(h2o_cache* cache, int low_bits, int hi_bits);

/* The digit layout in use: digits[0] low_bits, [1] hi_bits, [2] levels
 * (digits of the largest rank), [3] table entries; all 0 when rolling is
 * off.  digits: int32[4], host memory. */
H2O_API int h2o_cache_rolling_digits(const h2o_cache* cache, int32_t* digits);

/* Static sparse pattern combined with heavy hitters ("... 深度解读报告",
 * section 4.5, Table 2: Sparse Transformer strided / fixed patterns plus H2).
 * Positions offset, offset + stride, ..., offset + (count - 1) * stride are
 * kept for good: h2o_prefill keeps those below L - recent before choosing
 * heavy hitters, and h2o_decode_step never evicts them (they are not
 * eviction candidates once outside the recent window).  They occupy
 * heavy-budget slots, so count <= heavy; the heavy hitters fill the remaining
 * heavy slots.  offset 0 and stride s give the strided lattice 0, s, 2s, ...;
 * offset l - 1 and stride l the fixed pattern's block-summary positions (the
 * last position of each block of l); stride 1 the first `count` tokens.
 * count = 0 (the default) turns it off.  Host-side and immediate: it applies
 * to the prefill and decode calls made after it.  It is configuration, not
 * state: export/import do not carry it.  Returns H2O_EINVAL for offset < 0,
 * stride < 1, count < 0, count > heavy, or a last position beyond int32. */
H2O_API int h2o_cache_set_static_pattern(h2o_cache* cache, int offset, int stride, int count);

/* info[0..9] = {batch, heads, head_dim, heavy, recent, kv_dtype,
 *               decode splits in use (-1: warp per pair), decode stages in
 *               use, decode threads per CTA, 0}. */
H2O_API int h2o_cache_info(const h2o_cache* cache, int32_t* info);

/* Column sums of the prefill without any device allocation.  The paper has
 * no counterpart: this exists for callers that cannot call cudaMalloc, such
 * as engines that hand out all device memory from their own pools and forbid
 * allocation after start-up, or loops that cannot afford the device-wide
 * synchronisation a cudaMalloc implies.  It runs the same kernels as
 * h2o_prefill_ex without an attention output and returns the same values,
 * bit for bit, as that call's colsum_or_null (with an attention output,
 * h2o_prefill_ex takes its column sums from the output pass instead, and
 * they agree within 1e-5 relative):
 *   colsum[b,h,j] = sum_{i>=j} softmax_i(scale * q_i . k_j)    (causal rows)
 * q, k: [B, H, L, D] device pointers in kv_dtype (16-byte aligned); colsum:
 * [B, H, L] float32 device output.  No cache is involved and nothing is kept.
 * The per-row log-sum-exp scratch lives in a fixed array inside the library
 * (8 MiB, held on every GPU that loads the library until the process exits),
 * so B*H*L must be <= 2,097,152; larger sizes return H2O_EINVAL before any
 * launch.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Every call shares the one array: calls whose
 * kernels overlap on the GPU (different streams, or several host threads)
 * race and corrupt each other's results, so serialise them.  Each call
 * writes every scratch entry it reads, so stale contents from a previous
 * call do no harm, unless one of the call's bounded device waits gave up:
 * the call then leaves some entries unwritten and latches an error word
 * (also a fixed library array, cleared with cudaMemsetAsync at the start of
 * every call) that h2o_prefill_colsum_static_check reports.  Asynchronous
 * on `stream`. */
H2O_API int h2o_prefill_colsum_static(const void* q, const void* k, int batch, int heads, int head_dim,
                                      int prompt_len, int kv_dtype, float scale, float* colsum, void* stream);

/* Synchronous.  Wait for `stream`, then report H2O_EDEVICE if the kernels of
 * the last h2o_prefill_colsum_static call on the current device latched a
 * device error (its column sums are then not valid), else H2O_OK.  Allocates
 * nothing.  Call it on the stream of that call, before the next one. */
H2O_API int h2o_prefill_colsum_static_check(void* stream);

/* Self-test of the bounded waits every kernel of the library uses (they are
 * how a device-side stall becomes an H2O_EDEVICE status instead of a hang).
 * Launches one warp that waits, `polls` times (each poll suspends at most
 * about 1 us), on an mbarrier nothing arrives at: once with the CTA-scope
 * wait the stage rings use, once with the cluster-scope wait the decode
 * cluster exchange uses.  Synchronous.  On return gave_up[0] and gave_up[1]
 * are 1 if the respective wait gave up (the expected result) and elapsed_ns
 * holds the device time the two waits took together.  polls must be in
 * 1..1000000 (at most about 2 s); other values return H2O_EINVAL.  The device
 * stays usable afterwards: nothing is left waiting. */
H2O_API int h2o_selftest_wait_timeout(unsigned polls, int* gave_up, unsigned long long* elapsed_ns);

/* Fault injection for tests of the callers' error paths: after `after`
 * more successful device allocations made by this library (from any
 * thread), the next one fails as if the device were out of memory (the call
 * that makes it returns H2O_ENOMEM and frees what it had allocated), and the
 * hook disarms itself.  after = -1 disarms it.  Host-side only: no kernel
 * and no device is involved.  Returns H2O_EINVAL for after < -1. */
H2O_API int h2o_debug_fail_alloc(int after);

/* Thread-local message describing the last error returned on this thread. */
H2O_API const char* h2o_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* H2O_GB300_H */
