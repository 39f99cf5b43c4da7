// Internal definitions shared by the C-ABI layer and the kernels.
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace h2o {

// Device error bits latched in h2o_cache::err (reported by h2o_cache_check).
enum : int {
  ERR_MBAR_TIMEOUT = 1,  // a consumer's wait for a filled stage gave up
  ERR_NO_CANDIDATE = 2,  // full cache but no slot outside the recent window
  ERR_SELECT = 4,        // prefill selection did not find `heavy` keys
  ERR_RING_TIMEOUT = 8,  // the producer's wait for a free stage gave up
  ERR_MMA_TIMEOUT = 16,  // a prefill wait for tensor-core results gave up
  ERR_XCH_TIMEOUT = 32,  // a wait for the partial results a peer CTA pushes gave up
};

// Static sparse pattern combined with heavy hitters ("H2O ... 深度解读报告",
// section 4.5, Table 2): positions offset, offset + stride, ...,
// offset + (count - 1) * stride are kept for good.  They take heavy-budget
// slots (count <= heavy), the prefill keeps them first and decode never
// evicts them.  count = 0: no pattern.
struct StaticPattern {
  int offset;
  int stride;
  int count;
};

__host__ __device__ __forceinline__ bool is_protected(const StaticPattern& sp, int pos) {
  if (sp.count <= 0) return false;
  const int d = pos - sp.offset;
  if (d < 0) return false;
  const int k = d / sp.stride;
  return k < sp.count && k * sp.stride == d;
}

// Position rolling: a rank r is split into digits, the lowest of `low` bits
// and digits of `hi` bits above it; level l's digit selects one entry of that
// level's rotation table.  rope_levels_for: the digits every rank
// 0..max_rank needs; rope_entries_for: the table entries they take (2^low on
// level 0, 2^hi on the levels between, and only as many as the top digit
// reaches on the top level).  rope_entry: the entry of level l's digit of r.
__host__ __device__ __forceinline__ int rope_levels_for(int max_rank, int low, int hi) {
  int l = 1;
  while (l < 6 && (1LL << (low + hi * (l - 1))) <= max_rank) ++l;
  return l;
}
__host__ __device__ __forceinline__ int rope_entries_for(int max_rank, int low, int hi) {
  const int l = rope_levels_for(max_rank, low, hi);
  if (l == 1) return max_rank + 1;
  return (1 << low) + (1 << hi) * (l - 2) + (max_rank >> (low + hi * (l - 2))) + 1;
}
__host__ __device__ __forceinline__ int rope_entry(int r, int l, int low, int hi) {
  return l == 0 ? (r & ((1 << low) - 1))
                : (1 << low) + (1 << hi) * (l - 1) + ((r >> (low + hi * (l - 1))) & ((1 << hi) - 1));
}
// digit widths the kernel takes: low 4..6 bits, hi 4..6 bits
constexpr int kRopeMinBits = 4, kRopeMaxBits = 6;

// Per-pair counters kept on the device so decode steps can be replayed from
// a CUDA graph: next absolute position, occupied slots, ring head.
struct PairCtr {
  int p;
  int count;
  int head;
  int pad;
};

struct DecodeParams {
  void* K;            // [P, C, D] slot store, kv dtype
  void* V;            // [P, C, D]
  float* score;       // [P, C] accumulated attention
  int* pos;           // [P, C] absolute position per slot, -1 = empty
  int* ring;          // [P, R] slot ids of the recent window
  PairCtr* ctr;       // [P]
  const void* q;      // [P, D]
  const void* k_new;  // [P, D]
  const void* v_new;  // [P, D]
  float* out;         // [P, D]
  int* evicted;       // [P] or nullptr
  int* err;
  int C, R;
  int chunk;          // slots per CTA of a pair's cluster (multiple of 4)
  float qscale;       // scale * log2(e): logits kept in the base-2 domain
  int nstage;         // stage ring depth: a multiple of the cluster kernel's consumer warps (<= 18), or 2..8 per warp (warp per pair)
  int prefetch;       // 1: the previous kernel on the stream did not touch
                      // this cache, so its slot store may be read before the
                      // grid-dependency wait
  int pairs;          // P
  // position rolling (rotary embedding at positions inside the cache), or
  // both nullptr: the rank of each slot among the kept tokens in text order,
  // and the rotation tables of the ranks' digits: entry rope_entry(., l, low,
  // hi) of digit d holds cos and sin of d * (weight of level l) *
  // base^(-2i/D), level 0 weighing 1 and level l 2^(low + hi(l-1)), for every
  // pair i < D/2, in lane order (float4 h * LPR + g holds the cosines, then
  // the sines, of pairs g * EPV/2 + 2h and + 2h + 1, where a row's LPR lanes
  // take EPV elements each), so that the lanes of a row read consecutive
  // 16-byte words
  int* rank;           // [P, C]
  const float2* rope;  // [rope_entries_for(C, rope_low_bits, rope_hi_bits), D / 2]
  int rope_levels;     // digits of the largest rank, C (rope_levels_for)
  int rope_low_bits;   // bits of the lowest digit
  int rope_hi_bits;    // bits of each digit above it
  StaticPattern sp;    // protected positions, never eviction candidates
#ifdef H2O_DECODE_TIMELINE
  int tl_slot;  // profiling build: which stamp buffer this launch writes
#endif
};

#ifdef H2O_DECODE_TIMELINE
// Profiling build only (compiled with -DH2O_DECODE_TIMELINE): every CTA of a
// cluster-kernel decode launch records %globaltimer at kTimelineStamps fixed
// points into buffer tl_slot of a device array; launches take the buffers
// in turn, so the last kTimelineSlots launches can be read back.
constexpr int kTimelineSlots = 4;
constexpr int kTimelineMaxCtas = 4096;
constexpr int kTimelineStamps = 11;
cudaError_t decode_timeline_read(void* dst, size_t bytes);
#endif

struct PrefillParams {
  const void* q;  // [P, L, D]
  const void* k;
  const void* v;
  float* out;     // [P, L, D] or nullptr
  float* lse2;    // [P, L] log2-domain row log-sum-exp of the scaled logits
  float* colsum;  // [P, L]
  int L;          // row stride of the [P, L, D] inputs and [P, L] outputs (the longest prompt)
  float qscale;   // scale * log2(e)
  int* err = nullptr;  // device error bits, or nullptr
  const int* lens = nullptr;  // [B] per-batch-row prompt lengths (device), or nullptr: all L
  int heads = 1;              // pairs per batch row (maps a pair to its length)
  // When the output pass runs: column-sum partials it writes, one 128-float
  // row per (query block qb, key block kb <= qb, TMEM lane quarter), reduced
  // into colsum afterwards; nullptr: the column pass computes colsum.
  float* cs_part = nullptr;
};
// Floats of the column-sum partials for prompts of L rows (stride) and P pairs.
__host__ __device__ inline size_t colsum_partial_floats(int L, int P) {
  const size_t nb = (static_cast<size_t>(L) + 127) / 128;
  return static_cast<size_t>(P) * (nb * (nb + 1) / 2) * 4 * 128;
}

struct SelectParams {
  const void* k;         // prompt keys   [P, L, D]
  const void* v;         // prompt values [P, L, D]
  const float* colsum;   // [P, L]
  void* K;               // slot store [P, C, D]
  void* V;
  float* score;
  int* pos;
  int* ring;
  PairCtr* ctr;
  int* err;
  int L, heavy, recent, C;    // L: row stride of the inputs (the longest prompt)
  const int* lens = nullptr;  // [B] per-batch-row prompt lengths (device), or nullptr: all L
  int heads = 1;
  StaticPattern sp = {0, 1, 0};  // protected positions: kept before any heavy hitter
};

// Prompt length of pair `pair`: its batch row's length, clamped to [0, L],
// when lengths are given, else L.  Read after the grid-dependency wait (the
// lengths may come from an earlier kernel).
__device__ __forceinline__ int pair_len(const int* lens, int heads, int L, int pair) {
  if (!lens) return L;
  const int n = lens[pair / heads];
  return n < 0 ? 0 : (n > L ? L : n);
}

// Record the thread-local message returned by h2o_last_error(); returns code.
int set_error(int code, const char* fmt, ...);

// Raise a kernel's dynamic shared-memory limit (and optionally allow
// non-portable cluster sizes) once per process and device; later calls with
// a smaller or equal size do nothing, so launches inside stream capture make
// no attribute calls.
cudaError_t kernel_attrs(const void* kern, size_t smem_bytes, bool nonportable_cluster);

// Launchers (return the launch error; they do not synchronise).
cudaError_t launch_decode(const DecodeParams& prm, int dtype, int D, int pairs, int splits, cudaStream_t s);
// splits value selecting the warp-per-pair decode kernel (one warp streams
// a whole pair, each CTA's warps work through several pairs in turn)
constexpr int kDecodeWarpPerPair = -1;
struct DecodeShape {
  int splits;  // CTAs (one cluster) per pair, or kDecodeWarpPerPair
  int stages;  // shared-memory ring depth per CTA (per warp in warp-per-pair mode)
};
// rope_entries: position rolling's rotation-table entries (cluster kernel
// only, one more int of shared memory per slot), 0 when off
DecodeShape decode_pick_shape(int dtype, int D, int pairs, int C, int rope_entries = 0);
// Position rolling's digit widths for a shape: the fewest levels whose
// tables still leave the automatic launch shape as many resident CTAs as the
// smallest tables do, then the fewest entries.
struct RopeRadix {
  int low, hi;
};
RopeRadix decode_pick_rope_radix(int dtype, int D, int pairs, int C);
// CTAs of this shape that fit on the device at once (0: cannot launch);
// rope_entries: position rolling's rotation-table entries, 0 when off
int decode_resident(int dtype, int D, int splits, int nstage, int chunk, int pairs, int rope_entries = 0);
int decode_chunk(int C, int splits);
int decode_max_stages();
int decode_stage_multiple(int splits, bool rope = false);  // ring depths for this cluster size must be multiples of this
int decode_max_chunk();
int decode_threads(int splits, bool rope = false);  // threads per CTA of the cluster kernel
// warp-per-pair kernel: limits, and whether a shape can run (0 = no)
int decode_warp_max_slots();
int decode_warp_min_stages();
int decode_warp_max_stages();
int decode_warp_resident(int dtype, int D, int nstage, int C);
int decode_warp_default_stages(int dtype, int D, int C, int pairs);

cudaError_t launch_prefill_stats(const PrefillParams& prm, int dtype, int D, int pairs, cudaStream_t s);
cudaError_t launch_prefill_colsum(const PrefillParams& prm, int dtype, int D, int pairs, cudaStream_t s);
// colsum from the output pass's partials (prm.cs_part)
cudaError_t launch_colsum_reduce(const PrefillParams& prm, int pairs, cudaStream_t s);
// fp16 passes on tcgen05 (row statistics without the attention output)
cudaError_t launch_prefill_stats_tc(const PrefillParams& prm, int D, int pairs, cudaStream_t s);
cudaError_t launch_prefill_colsum_tc(const PrefillParams& prm, int D, int pairs, cudaStream_t s);
cudaError_t launch_prefill_select(const SelectParams& prm, int dtype, int D, int pairs, cudaStream_t s);
cudaError_t launch_reset(PairCtr* ctr, int* pos, float* score, int* ring, int pairs, int C, int R,
                         cudaStream_t s);
// lse (natural log) from the log2-domain buffer, for callers that ask for it
cudaError_t launch_lse_export(const float* lse2, float* lse, size_t n, cudaStream_t s);

}  // namespace h2o

// The opaque cache object behind the C ABI.
struct h2o_cache {
  int B, H, D, heavy, recent, C, dtype, elem, P;
  void* K;
  void* V;
  float* score;
  int* pos;
  int* ring;
  h2o::PairCtr* ctr;
  int* err;
  // prefill workspace, grown on demand: lse2 and colsum, [P, ws_len] each
  float* ws;
  size_t ws_len;
  // column-sum partials of the output pass (colsum_partial_floats), grown on demand
  float* wsp;
  size_t wsp_len;
  int device, num_sms;
  int splits_override, stages_override;
  h2o::DecodeShape shape_auto;
  long long host_next_p;  // host mirror of the next position (overflow check)
  // position rolling: slot ranks [P, C] and the digit rotation tables
  // [rope_entries_for(C, rope_low, rope_hi), D/2]; nullptr when off
  int* rank;
  float2* rope;
  float rope_base;
  int rope_low, rope_hi;  // the ranks' digit widths (decode_pick_rope_radix)
  h2o::StaticPattern sp;  // static sparse pattern (count 0: none)
};
