// C ABI of the H2O library: cache object, argument checks, error reporting and
// stream-ordered launches of the decode / prefill kernels.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <map>
#include <mutex>
#include <utility>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "h2o.h"
#include "h2o_internal.cuh"
#include "ptx.cuh"

namespace {
// Position rolling: the rank of every kept slot among its pair's kept tokens
// in text order (-1 for an empty slot).  pos: [P, C] host array.
void ranks_from_positions(const int* pos, int P, int C, std::vector<int>& out) {
  out.assign(static_cast<size_t>(P) * C, -1);
  std::vector<std::pair<int, int>> kept;
  kept.reserve(C);
  for (int i = 0; i < P; ++i) {
    kept.clear();
    for (int j = 0; j < C; ++j) {
      const int x = pos[static_cast<size_t>(i) * C + j];
      if (x >= 0) kept.emplace_back(x, j);
    }
    std::sort(kept.begin(), kept.end());
    for (size_t r = 0; r < kept.size(); ++r) out[static_cast<size_t>(i) * C + kept[r].second] = static_cast<int>(r);
  }
}


thread_local char g_msg[512] = "";

// NVTX range around an ABI call (visible in Nsight Systems / Compute; a
// no-op when no tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

#ifdef H2O_DECODE_TIMELINE
// Profiling build: the stamp buffer the next decode launch writes.
std::atomic<long long> g_tl_next{0};
#endif

// Allocation-failure injection (h2o_debug_fail_alloc): the number of device
// allocations still allowed before the next one fails, or -1 when disarmed.
std::atomic<long long> g_alloc_budget{-1};

// Every device allocation of the library goes through here.
cudaError_t dev_alloc(void** p, size_t bytes) {
  long long b = g_alloc_budget.load();
  while (b >= 0) {
    if (g_alloc_budget.compare_exchange_weak(b, b - 1)) {
      if (b == 0) {  // this is the allocation that fails; the hook disarms
        *p = nullptr;
        return cudaErrorMemoryAllocation;
      }
      break;
    }
  }
  return cudaMalloc(p, bytes);
}
template <typename T>
cudaError_t dev_alloc(T** p, size_t bytes) {
  void* v = nullptr;
  cudaError_t e = dev_alloc(&v, bytes);
  *p = static_cast<T*>(v);
  return e;
}

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(e == cudaErrorMemoryAllocation ? H2O_ENOMEM : H2O_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e),
              cudaGetErrorString(e));
}

constexpr int kHeaderInts = 16;
constexpr int kMagic = 0x48324F31;
constexpr int kMaxSlots = 65536;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t kv_bytes(const h2o_cache* c) { return static_cast<size_t>(c->P) * c->C * c->D * c->elem; }

int chunk_for(int C, int splits) { return h2o::decode_chunk(C, splits); }

// Which cache the last library kernel issued on each stream worked on.  A
// decode step may read its slot store before the programmatic
// grid-dependency wait only if the kernel just before it on the stream did not
// touch the same cache (every library kernel issues its launch-dependents
// trigger after its own wait, so all earlier kernels are complete by then).
std::mutex g_stream_mu;
std::map<const void*, const h2o_cache*> g_last_on_stream;

bool touch_stream(const h2o_cache* c, void* stream) {
  std::lock_guard<std::mutex> lock(g_stream_mu);
  auto it = g_last_on_stream.find(stream);
  const bool other = it == g_last_on_stream.end() || it->second != c;
  g_last_on_stream[stream] = c;
  return other;
}

void forget_cache(const h2o_cache* c) {
  std::lock_guard<std::mutex> lock(g_stream_mu);
  for (auto it = g_last_on_stream.begin(); it != g_last_on_stream.end();)
    it = it->second == c ? g_last_on_stream.erase(it) : std::next(it);
}

int splits_in_use(const h2o_cache* c) {
  return c->splits_override != 0 ? c->splits_override : c->shape_auto.splits;
}
int stages_in_use(const h2o_cache* c) {
  return c->stages_override > 0 ? c->stages_override : c->shape_auto.stages;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

namespace h2o {
int set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

cudaError_t kernel_attrs(const void* kern, size_t smem_bytes, bool nonportable_cluster) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, size_t> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  auto key = std::make_pair(kern, dev);
  auto it = done.find(key);
  if (it != done.end() && it->second >= smem_bytes) return cudaSuccess;
  if (smem_bytes > 48 * 1024 &&
      (e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_bytes))) !=
          cudaSuccess)
    return e;
  if (nonportable_cluster &&
      (e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
    return e;
  done[key] = smem_bytes;
  return cudaSuccess;
}
}  // namespace h2o

namespace {
// One warp; lane 0 waits on an mbarrier that no thread or copy will ever
// complete, first with the CTA-scope bounded wait, then with the
// cluster-scope one, and records whether each gave up.
__global__ void wait_timeout_probe(unsigned polls, int* out, unsigned long long* ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  h2o::mbar_init(&bar, 1);
  h2o::fence_mbar_init();
  unsigned long long t0, t1;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  const bool a = h2o::mbar_wait_bounded(&bar, 0u, polls);
  const bool b = h2o::mbar_wait_cluster_bounded(&bar, 0u, polls);
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
  out[0] = a ? 0 : 1;
  out[1] = b ? 0 : 1;
  *ns = t1 - t0;
}
}  // namespace

extern "C" {

const char* h2o_last_error(void) { return g_msg; }

int h2o_cache_create(int batch, int heads, int head_dim, int heavy_budget, int recent_budget, int kv_dtype,
                     h2o_cache** out) {
  NvtxRange nvtx("h2o_cache_create");
  if (!out) return fail(H2O_EINVAL, "h2o_cache_create: out is NULL");
  *out = nullptr;
  if (batch < 1 || heads < 1) return fail(H2O_EINVAL, "h2o_cache_create: batch and heads must be >= 1");
  if (head_dim != 64 && head_dim != 128) return fail(H2O_EINVAL, "h2o_cache_create: head_dim must be 64 or 128");
  if (heavy_budget < 0) return fail(H2O_EINVAL, "h2o_cache_create: heavy_budget must be >= 0");
  if (recent_budget < 1) return fail(H2O_EINVAL, "h2o_cache_create: recent_budget must be >= 1");
  if (kv_dtype != H2O_F16 && kv_dtype != H2O_F32) return fail(H2O_EINVAL, "h2o_cache_create: bad kv_dtype");
  const long long C = static_cast<long long>(heavy_budget) + recent_budget;
  if (C > kMaxSlots) return fail(H2O_EINVAL, "h2o_cache_create: heavy+recent must be <= %d", kMaxSlots);
  const long long P = static_cast<long long>(batch) * heads;
  if (P > 65535) return fail(H2O_EINVAL, "h2o_cache_create: batch*heads must be <= 65535");

  h2o_cache* c = new (std::nothrow) h2o_cache();
  if (!c) return fail(H2O_ENOMEM, "h2o_cache_create: host allocation failed");
  std::memset(c, 0, sizeof(*c));
  c->B = batch;
  c->H = heads;
  c->D = head_dim;
  c->heavy = heavy_budget;
  c->recent = recent_budget;
  c->C = static_cast<int>(C);
  c->dtype = kv_dtype;
  c->elem = kv_dtype == H2O_F16 ? 2 : 4;
  c->P = static_cast<int>(P);
  c->sp = h2o::StaticPattern{0, 1, 0};
  cudaError_t e = cudaGetDevice(&c->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
  if (e != cudaSuccess) {
    delete c;
    return cuda_fail(e, "h2o_cache_create: no CUDA device");
  }
  const size_t nslot = static_cast<size_t>(c->P) * c->C;
  const size_t nring = static_cast<size_t>(c->P) * c->recent;
  if ((e = dev_alloc(&c->K, kv_bytes(c))) != cudaSuccess || (e = dev_alloc(&c->V, kv_bytes(c))) != cudaSuccess ||
      (e = dev_alloc(&c->score, nslot * sizeof(float))) != cudaSuccess ||
      (e = dev_alloc(&c->pos, nslot * sizeof(int))) != cudaSuccess ||
      (e = dev_alloc(&c->ring, nring * sizeof(int))) != cudaSuccess ||
      (e = dev_alloc(&c->ctr, static_cast<size_t>(c->P) * sizeof(h2o::PairCtr))) != cudaSuccess ||
      (e = dev_alloc(&c->err, sizeof(int))) != cudaSuccess) {
    h2o_cache_destroy(c);
    return cuda_fail(e, "h2o_cache_create: cudaMalloc");
  }
  if ((e = cudaMemset(c->K, 0, kv_bytes(c))) != cudaSuccess || (e = cudaMemset(c->V, 0, kv_bytes(c))) != cudaSuccess ||
      (e = cudaMemset(c->score, 0, nslot * sizeof(float))) != cudaSuccess ||
      (e = cudaMemset(c->pos, 0xff, nslot * sizeof(int))) != cudaSuccess ||
      (e = cudaMemset(c->ring, 0xff, nring * sizeof(int))) != cudaSuccess ||
      (e = cudaMemset(c->ctr, 0, static_cast<size_t>(c->P) * sizeof(h2o::PairCtr))) != cudaSuccess ||
      (e = cudaMemset(c->err, 0, sizeof(int))) != cudaSuccess || (e = cudaDeviceSynchronize()) != cudaSuccess) {
    h2o_cache_destroy(c);
    return cuda_fail(e, "h2o_cache_create: initialisation");
  }
  // cluster size: the largest that keeps every CTA of the grid resident
  c->shape_auto = h2o::decode_pick_shape(c->dtype, c->D, c->P, c->C);
  *out = c;
  return H2O_OK;
}

void h2o_cache_destroy(h2o_cache* c) {
  if (!c) return;
  forget_cache(c);
  cudaFree(c->K);
  cudaFree(c->V);
  cudaFree(c->score);
  cudaFree(c->pos);
  cudaFree(c->ring);
  cudaFree(c->ctr);
  cudaFree(c->err);
  cudaFree(c->ws);
  cudaFree(c->wsp);
  cudaFree(c->rank);
  cudaFree(c->rope);
  delete c;
}

int h2o_cache_reset(h2o_cache* c, void* stream) {
  NvtxRange nvtx("h2o_cache_reset");
  if (!c) return fail(H2O_EINVAL, "h2o_cache_reset: cache is NULL");
  touch_stream(c, stream);
  cudaError_t e = h2o::launch_reset(c->ctr, c->pos, c->score, c->ring, c->P, c->C, c->recent, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "h2o_cache_reset");
  c->host_next_p = 0;
  return H2O_OK;
}

// The prefill for a prompt of prompt_len rows per pair, or, with lens, of
// lens[b] rows for batch row b (prompt_len then being the row stride).
static int prefill_impl(h2o_cache* c, const void* q, const void* k, const void* v, int prompt_len,
                        const int32_t* lens, float scale, float* out_or_null, float* colsum_or_null,
                        float* lse_or_null, void* stream) {
  NvtxRange nvtx("h2o_prefill");
  if (!c) return fail(H2O_EINVAL, "h2o_prefill: cache is NULL");
  if (prompt_len < 0) return fail(H2O_EINVAL, "h2o_prefill: prompt_len must be >= 0");
  if (prompt_len == 0) return h2o_cache_reset(c, stream);
  if (c->rope)
    return fail(H2O_ESTATE, "h2o_prefill: position rolling is on and the prefill applies no rotary embedding "
                            "(decode from an empty cache instead)");
  if (!q || !k || !v) return fail(H2O_EINVAL, "h2o_prefill: q, k and v are required");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || (out_or_null && !aligned16(out_or_null)))
    return fail(H2O_EINVAL, "h2o_prefill: device pointers must be 16-byte aligned");
  if (!(scale > 0.f) || scale != scale) return fail(H2O_EINVAL, "h2o_prefill: scale must be positive");
  const size_t need = static_cast<size_t>(prompt_len);
  cudaError_t e;
  if (need > c->ws_len) {
    // grow the workspace: [P, L] log2-domain lse + [P, L] column sums
    if (c->ws) {
      if ((e = cudaStreamSynchronize(as_stream(stream))) != cudaSuccess) return cuda_fail(e, "h2o_prefill: sync");
      cudaFree(c->ws);
      c->ws = nullptr;
      c->ws_len = 0;
    }
    if ((e = dev_alloc(&c->ws, 2 * need * c->P * sizeof(float))) != cudaSuccess)
      return cuda_fail(e, "h2o_prefill: workspace cudaMalloc");
    c->ws_len = need;
  }
  // with the attention output on the tensor-core path, the output pass also
  // produces the column sums, through a partials workspace that grows with
  // the square of the prompt; beyond 2 GB the column pass runs instead
  size_t need_p = (out_or_null && c->dtype == H2O_F16) ? h2o::colsum_partial_floats(prompt_len, c->P) : 0;
  if (need_p * sizeof(float) > (static_cast<size_t>(2) << 30)) need_p = 0;
  if (need_p > c->wsp_len) {
    if (c->wsp) {
      if ((e = cudaStreamSynchronize(as_stream(stream))) != cudaSuccess) return cuda_fail(e, "h2o_prefill: sync");
      cudaFree(c->wsp);
      c->wsp = nullptr;
      c->wsp_len = 0;
    }
    if ((e = dev_alloc(&c->wsp, need_p * sizeof(float))) != cudaSuccess)
      return cuda_fail(e, "h2o_prefill: partials workspace cudaMalloc");
    c->wsp_len = need_p;
  }
  const size_t plen = static_cast<size_t>(c->P) * prompt_len;
  h2o::PrefillParams pp;
  pp.q = q;
  pp.k = k;
  pp.v = v;
  pp.out = out_or_null;
  pp.lse2 = c->ws;
  pp.colsum = colsum_or_null ? colsum_or_null : c->ws + plen;
  pp.L = prompt_len;
  pp.qscale = scale * 1.4426950408889634f;
  pp.err = c->err;
  pp.lens = lens;
  pp.heads = c->H;
  pp.cs_part = need_p ? c->wsp : nullptr;
  cudaStream_t s = as_stream(stream);
  touch_stream(c, stream);
  if ((e = h2o::launch_prefill_stats(pp, c->dtype, c->D, c->P, s)) != cudaSuccess)
    return cuda_fail(e, "h2o_prefill: row statistics launch");
  if ((e = h2o::launch_prefill_colsum(pp, c->dtype, c->D, c->P, s)) != cudaSuccess)
    return cuda_fail(e, "h2o_prefill: column sum launch");
  h2o::SelectParams sp;
  sp.k = k;
  sp.v = v;
  sp.colsum = pp.colsum;
  sp.K = c->K;
  sp.V = c->V;
  sp.score = c->score;
  sp.pos = c->pos;
  sp.ring = c->ring;
  sp.ctr = c->ctr;
  sp.err = c->err;
  sp.L = prompt_len;
  sp.heavy = c->heavy;
  sp.recent = c->recent;
  sp.C = c->C;
  sp.lens = lens;
  sp.heads = c->H;
  sp.sp = c->sp;
  if ((e = h2o::launch_prefill_select(sp, c->dtype, c->D, c->P, s)) != cudaSuccess)
    return cuda_fail(e, "h2o_prefill: select launch");
  if (lse_or_null && (e = h2o::launch_lse_export(pp.lse2, lse_or_null, plen, s)) != cudaSuccess)
    return cuda_fail(e, "h2o_prefill: lse export");
  c->host_next_p = prompt_len;  // an upper bound on every pair's next position
  return H2O_OK;
}

int h2o_prefill_ex(h2o_cache* c, const void* q, const void* k, const void* v, int prompt_len, float scale,
                   float* out_or_null, float* colsum_or_null, float* lse_or_null, void* stream) {
  return prefill_impl(c, q, k, v, prompt_len, nullptr, scale, out_or_null, colsum_or_null, lse_or_null, stream);
}

int h2o_prefill_ragged(h2o_cache* c, const void* q, const void* k, const void* v, int max_len,
                       const int32_t* lengths, float scale, float* out_or_null, float* colsum_or_null,
                       float* lse_or_null, void* stream) {
  if (!lengths || (reinterpret_cast<uintptr_t>(lengths) & 3u) != 0)
    return fail(H2O_EINVAL, "h2o_prefill_ragged: lengths must be a 4-byte aligned device pointer");
  return prefill_impl(c, q, k, v, max_len, lengths, scale, out_or_null, colsum_or_null, lse_or_null, stream);
}

int h2o_prefill(h2o_cache* c, const void* q, const void* k, const void* v, int prompt_len, float scale,
                float* out_or_null, void* stream) {
  return h2o_prefill_ex(c, q, k, v, prompt_len, scale, out_or_null, nullptr, nullptr, stream);
}

int h2o_decode_step(h2o_cache* c, const void* q, const void* k_new, const void* v_new, float scale, float* out,
                    int32_t* evicted_or_null, void* stream) {
  NvtxRange nvtx("h2o_decode_step");
  if (!c) return fail(H2O_EINVAL, "h2o_decode_step: cache is NULL");
  if (!q || !k_new || !v_new || !out) return fail(H2O_EINVAL, "h2o_decode_step: q, k_new, v_new and out are required");
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(out))
    return fail(H2O_EINVAL, "h2o_decode_step: device pointers must be 16-byte aligned");
  if (!(scale > 0.f) || scale != scale) return fail(H2O_EINVAL, "h2o_decode_step: scale must be positive");
  if (c->host_next_p >= INT_MAX) return fail(H2O_ESTATE, "h2o_decode_step: int32 positions exhausted");
  const int splits = splits_in_use(c);
  h2o::DecodeParams dp;
  dp.K = c->K;
  dp.V = c->V;
  dp.score = c->score;
  dp.pos = c->pos;
  dp.ring = c->ring;
  dp.ctr = c->ctr;
  dp.q = q;
  dp.k_new = k_new;
  dp.v_new = v_new;
  dp.out = out;
  dp.evicted = evicted_or_null;
  dp.err = c->err;
  dp.C = c->C;
  dp.R = c->recent;
  dp.chunk = chunk_for(c->C, splits);
  dp.nstage = stages_in_use(c);
  dp.qscale = scale * 1.4426950408889634f;
  dp.prefetch = touch_stream(c, stream) ? 1 : 0;
  dp.pairs = c->P;
  dp.rank = c->rank;
  dp.rope = c->rope;
  dp.rope_low_bits = c->rope_low;
  dp.rope_hi_bits = c->rope_hi;
  dp.rope_levels = c->rope ? h2o::rope_levels_for(c->C, c->rope_low, c->rope_hi) : 0;
  dp.sp = c->sp;
#ifdef H2O_DECODE_TIMELINE
  dp.tl_slot = static_cast<int>(g_tl_next.fetch_add(1) % h2o::kTimelineSlots);
#endif
  cudaError_t e = h2o::launch_decode(dp, c->dtype, c->D, c->P, splits, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "h2o_decode_step: launch");
  c->host_next_p += 1;
  return H2O_OK;
}

size_t h2o_cache_state_bytes(const h2o_cache* c) {
  if (!c) return 0;
  const size_t nslot = static_cast<size_t>(c->P) * c->C;
  return kHeaderInts * sizeof(int) + 2 * kv_bytes(c) + nslot * (sizeof(float) + sizeof(int)) +
         static_cast<size_t>(c->P) * c->recent * sizeof(int) + static_cast<size_t>(c->P) * sizeof(h2o::PairCtr);
}

int h2o_cache_export_state(const h2o_cache* c, void* host_buf, size_t bytes, void* stream) {
  NvtxRange nvtx("h2o_cache_export_state");
  if (!c || !host_buf) return fail(H2O_EINVAL, "h2o_cache_export_state: NULL argument");
  if (bytes < h2o_cache_state_bytes(c)) return fail(H2O_EINVAL, "h2o_cache_export_state: buffer too small");
  int* hdr = static_cast<int*>(host_buf);
  std::memset(hdr, 0, kHeaderInts * sizeof(int));
  hdr[0] = kMagic;
  hdr[1] = 1;
  hdr[2] = c->B;
  hdr[3] = c->H;
  hdr[4] = c->D;
  hdr[5] = c->heavy;
  hdr[6] = c->recent;
  hdr[7] = c->dtype;
  unsigned char* p = static_cast<unsigned char*>(host_buf) + kHeaderInts * sizeof(int);
  const size_t nslot = static_cast<size_t>(c->P) * c->C;
  cudaStream_t s = as_stream(stream);
  cudaError_t e;
  struct {
    const void* src;
    size_t n;
  } parts[] = {{c->K, kv_bytes(c)},
               {c->V, kv_bytes(c)},
               {c->score, nslot * sizeof(float)},
               {c->pos, nslot * sizeof(int)},
               {c->ring, static_cast<size_t>(c->P) * c->recent * sizeof(int)},
               {c->ctr, static_cast<size_t>(c->P) * sizeof(h2o::PairCtr)}};
  for (auto& part : parts) {
    if ((e = cudaMemcpyAsync(p, part.src, part.n, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
      return cuda_fail(e, "h2o_cache_export_state: copy");
    p += part.n;
  }
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "h2o_cache_export_state: sync");
  return H2O_OK;
}

int h2o_cache_import_state(h2o_cache* c, const void* host_buf, size_t bytes, void* stream) {
  NvtxRange nvtx("h2o_cache_import_state");
  if (!c || !host_buf) return fail(H2O_EINVAL, "h2o_cache_import_state: NULL argument");
  if (bytes < h2o_cache_state_bytes(c)) return fail(H2O_EINVAL, "h2o_cache_import_state: buffer too small");
  const int* hdr = static_cast<const int*>(host_buf);
  if (hdr[0] != kMagic || hdr[1] != 1 || hdr[2] != c->B || hdr[3] != c->H || hdr[4] != c->D ||
      hdr[5] != c->heavy || hdr[6] != c->recent || hdr[7] != c->dtype)
    return fail(H2O_EINVAL, "h2o_cache_import_state: header does not match this cache");
  const unsigned char* p = static_cast<const unsigned char*>(host_buf) + kHeaderInts * sizeof(int);
  const size_t nslot = static_cast<size_t>(c->P) * c->C;
  const size_t nring = static_cast<size_t>(c->P) * c->recent;
  // validate counters before they reach the device
  const h2o::PairCtr* ctr =
      reinterpret_cast<const h2o::PairCtr*>(p + 2 * kv_bytes(c) + nslot * 8 + nring * sizeof(int));
  long long maxp = 0;
  for (int i = 0; i < c->P; ++i) {
    if (ctr[i].count < 0 || ctr[i].count > c->C || ctr[i].head < 0 || ctr[i].head >= c->recent || ctr[i].p < 0 ||
        ctr[i].count > ctr[i].p)
      return fail(H2O_EINVAL, "h2o_cache_import_state: counters of pair %d out of range", i);
    if (ctr[i].p > maxp) maxp = ctr[i].p;
  }
  cudaStream_t s = as_stream(stream);
  touch_stream(c, stream);
  cudaError_t e;
  struct {
    void* dst;
    size_t n;
  } parts[] = {{c->K, kv_bytes(c)},         {c->V, kv_bytes(c)},
               {c->score, nslot * sizeof(float)}, {c->pos, nslot * sizeof(int)},
               {c->ring, nring * sizeof(int)},    {c->ctr, static_cast<size_t>(c->P) * sizeof(h2o::PairCtr)}};
  for (auto& part : parts) {
    if ((e = cudaMemcpyAsync(part.dst, p, part.n, cudaMemcpyHostToDevice, s)) != cudaSuccess)
      return cuda_fail(e, "h2o_cache_import_state: copy");
    p += part.n;
  }
  std::vector<int> ranks;  // position rolling: ranks follow from the imported positions
  if (c->rope) {
    const int* pos = reinterpret_cast<const int*>(static_cast<const unsigned char*>(host_buf) +
                                                  kHeaderInts * sizeof(int) + 2 * kv_bytes(c) + nslot * 4);
    ranks_from_positions(pos, c->P, c->C, ranks);
    if ((e = cudaMemcpyAsync(c->rank, ranks.data(), nslot * sizeof(int), cudaMemcpyHostToDevice, s)) != cudaSuccess)
      return cuda_fail(e, "h2o_cache_import_state: ranks");
  }
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "h2o_cache_import_state: sync");
  c->host_next_p = maxp;
  return H2O_OK;
}

int h2o_cache_check(h2o_cache* c, void* stream) {
  NvtxRange nvtx("h2o_cache_check");
  if (!c) return fail(H2O_EINVAL, "h2o_cache_check: cache is NULL");
  cudaError_t e = cudaStreamSynchronize(as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "h2o_cache_check: stream");
  int flags = 0;
  if ((e = cudaMemcpy(&flags, c->err, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "h2o_cache_check: read flag");
  if (flags) {
    cudaMemset(c->err, 0, sizeof(int));
    cudaDeviceSynchronize();
    return fail(H2O_EDEVICE, "h2o_cache_check: device check fired (flags 0x%x:%s%s%s%s%s%s)", flags,
                (flags & h2o::ERR_MBAR_TIMEOUT) ? " copy-wait-timeout" : "",
                (flags & h2o::ERR_NO_CANDIDATE) ? " no-eviction-candidate" : "",
                (flags & h2o::ERR_SELECT) ? " prefill-select" : "",
                (flags & h2o::ERR_RING_TIMEOUT) ? " ring-wait-timeout" : "",
                (flags & h2o::ERR_MMA_TIMEOUT) ? " tensor-core-wait-timeout" : "",
                (flags & h2o::ERR_XCH_TIMEOUT) ? " cluster-exchange-timeout" : "");
  }
  return H2O_OK;
}

int h2o_cache_set_decode_shape(h2o_cache* c, int splits, int stages) {
  if (!c) return fail(H2O_EINVAL, "h2o_cache_set_decode_shape: cache is NULL");
  if (splits != 0 && splits != 1 && splits != 2 && splits != 4 && splits != 8 && splits != 16 &&
      splits != h2o::kDecodeWarpPerPair)
    return fail(H2O_EINVAL, "h2o_cache_set_decode_shape: splits must be 0, 1, 2, 4, 8, 16 or -1 (warp per pair)");
  const int s = splits != 0 ? splits : c->shape_auto.splits;
  int n = stages;
  if (n == 0) {
    if (s == c->shape_auto.splits)
      n = c->shape_auto.stages;
    else
      n = s == h2o::kDecodeWarpPerPair ? h2o::decode_warp_default_stages(c->dtype, c->D, c->C, c->P)
                                      : h2o::decode_stage_multiple(s, c->rope != nullptr);
  }
  if (s == h2o::kDecodeWarpPerPair) {
    if (c->rope)
      return fail(H2O_EINVAL, "h2o_cache_set_decode_shape: position rolling runs on the cluster kernel only");
    if (c->C > h2o::decode_warp_max_slots())
      return fail(H2O_EINVAL, "h2o_cache_set_decode_shape: warp per pair takes at most %d slots per pair",
                  h2o::decode_warp_max_slots());
    if (n < h2o::decode_warp_min_stages() || n > h2o::decode_warp_max_stages())
      return fail(H2O_EINVAL, "h2o_cache_set_decode_shape: warp per pair takes %d..%d stages",
                  h2o::decode_warp_min_stages(), h2o::decode_warp_max_stages());
    if (h2o::decode_warp_resident(c->dtype, c->D, n, c->C) <= 0)
      return fail(H2O_EINVAL, "h2o_cache_set_decode_shape: warp per pair with %d stages cannot be scheduled", n);
  } else {
    if (n < 0 || n > h2o::decode_max_stages() || n % h2o::decode_stage_multiple(s, c->rope != nullptr) != 0)
      return fail(H2O_EINVAL, "h2o_cache_set_decode_shape: stages must be a multiple of %d in 0..%d",
                  h2o::decode_stage_multiple(s, c->rope != nullptr), h2o::decode_max_stages());
    if (chunk_for(c->C, s) > h2o::decode_max_chunk())
      return fail(H2O_EINVAL, "h2o_cache_set_decode_shape: %d splits leave more than %d slots per CTA", s,
                  h2o::decode_max_chunk());
    if (h2o::decode_resident(c->dtype, c->D, s, n, chunk_for(c->C, s), c->P,
                             c->rope ? h2o::rope_entries_for(c->C, c->rope_low, c->rope_hi) : 0) < s)
      return fail(H2O_EINVAL, "h2o_cache_set_decode_shape: %d CTAs per pair with %d stages cannot be scheduled", s,
                  n);
  }
  c->splits_override = splits;
  c->stages_override = (splits == 0 && stages == 0) ? 0 : n;
  return H2O_OK;
}

int h2o_cache_set_static_pattern(h2o_cache* c, int offset, int stride, int count) {
  if (!c) return fail(H2O_EINVAL, "h2o_cache_set_static_pattern: cache is NULL");
  if (offset < 0 || stride < 1 || count < 0)
    return fail(H2O_EINVAL, "h2o_cache_set_static_pattern: need offset >= 0, stride >= 1, count >= 0");
  if (count > c->heavy)
    return fail(H2O_EINVAL, "h2o_cache_set_static_pattern: count %d exceeds the heavy budget %d", count, c->heavy);
  if (count > 0 && static_cast<long long>(offset) + static_cast<long long>(count - 1) * stride > INT_MAX)
    return fail(H2O_EINVAL, "h2o_cache_set_static_pattern: pattern positions exceed int32");
  c->sp = h2o::StaticPattern{offset, stride, count};
  return H2O_OK;
}

int h2o_cache_info(const h2o_cache* c, int32_t* info) {
  if (!c || !info) return fail(H2O_EINVAL, "h2o_cache_info: NULL argument");
  info[0] = c->B;
  info[1] = c->H;
  info[2] = c->D;
  info[3] = c->heavy;
  info[4] = c->recent;
  info[5] = c->dtype;
  info[6] = splits_in_use(c);
  info[7] = stages_in_use(c);
  info[8] = splits_in_use(c) == h2o::kDecodeWarpPerPair ? 128 : h2o::decode_threads(splits_in_use(c), c->rope != nullptr);
  info[9] = 0;
  return H2O_OK;
}

namespace {
// Position rolling on with this base and these digit widths (0, 0: the
// automatic ones), or off (base 0): ranks from the positions, rotation
// tables, launch shape.  `who` names the calling entry point in errors.
int set_rolling(h2o_cache* c, float rope_base, int low_req, int hi_req, const char* who) {
  char what_buf[160];
  auto what = [&](const char* step) {
    snprintf(what_buf, sizeof(what_buf), "%s: %s", who, step);
    return what_buf;
  };
  cudaError_t e = cudaDeviceSynchronize();  // the positions are read back below
  if (e != cudaSuccess) return cuda_fail(e, what("synchronise"));
  if (rope_base == 0.f) {
    cudaFree(c->rank);
    cudaFree(c->rope);
    c->rank = nullptr;
    c->rope = nullptr;
    c->rope_base = 0.f;
    // the plain kernel's own launch shape: an explicit one set for rolling
    // (ring depths in multiples of its consumer warps) goes back to automatic
    c->shape_auto = h2o::decode_pick_shape(c->dtype, c->D, c->P, c->C, 0);
    c->splits_override = 0;
    c->stages_override = 0;
    return H2O_OK;
  }
  const size_t nslot = static_cast<size_t>(c->P) * c->C;
  const h2o::RopeRadix radix = low_req > 0 ? h2o::RopeRadix{low_req, hi_req}
                                           : h2o::decode_pick_rope_radix(c->dtype, c->D, c->P, c->C);
  const int low = radix.low, hi = radix.hi;                  // bits of the ranks' lowest digit, of the others
  const int levels = h2o::rope_levels_for(c->C, low, hi);    // digits of the ranks 0..C
  const int entries = h2o::rope_entries_for(c->C, low, hi);  // table entries those digits take
  const size_t ntab = static_cast<size_t>(entries) * (c->D / 2);
  // Everything is built into new buffers and swapped in only once it is
  // complete, so a failure leaves the cache exactly as it was.
  int* rank = nullptr;
  float2* rope = nullptr;
  auto give_up = [&](cudaError_t err, const char* step) {
    cudaFree(rank);
    cudaFree(rope);
    return cuda_fail(err, what(step));
  };
  if ((e = dev_alloc(&rank, nslot * sizeof(int))) != cudaSuccess ||
      (e = dev_alloc(&rope, ntab * sizeof(float2))) != cudaSuccess)
    return give_up(e, "cudaMalloc");
  // rotation tables of the ranks' digits: the entry of level l's digit d
  // (h2o::rope_entry) holds, for every pair i, cos and sin of
  // d * w_l * base^(-2i/D), w_0 = 1 and w_l = 2^(low + hi(l-1)), computed in
  // double and stored as float in the order the decode lanes read them: a
  // row's LPR lanes take EPV elements (EPV / 2 pairs) each, and float4
  // h * LPR + g of an entry holds lane g's pairs 2h and 2h + 1 as
  // (cos, cos, sin, sin)
  const int epv = 16 / c->elem, lpr = c->D * c->elem / 16;
  std::vector<float2> tab(ntab);
  for (int e = 0; e < entries; ++e) {
    int lv = 0, d = e;  // level and digit of entry e
    if (levels > 1 && e >= (1 << low)) {
      lv = 1 + (e - (1 << low)) / (1 << hi);
      d = (e - (1 << low)) % (1 << hi);
    }
    const double w = lv == 0 ? 1.0 : std::ldexp(1.0, low + hi * (lv - 1));
    for (int i = 0; i < c->D / 2; ++i) {
      const double ang = d * w * std::pow(static_cast<double>(rope_base), -2.0 * i / c->D);
      const int g = i / (epv / 2), h = (i % (epv / 2)) / 2, x = i % 2;  // lane, float4 of the lane, pair in it
      float* f4 = reinterpret_cast<float*>(tab.data() + static_cast<size_t>(e) * (c->D / 2)) +
                  (static_cast<size_t>(h) * lpr + g) * 4;
      f4[x] = static_cast<float>(std::cos(ang));
      f4[2 + x] = static_cast<float>(std::sin(ang));
    }
  }
  std::vector<int> pos(nslot), ranks;
  if ((e = cudaMemcpy(pos.data(), c->pos, nslot * sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return give_up(e, "read positions");
  ranks_from_positions(pos.data(), c->P, c->C, ranks);
  if ((e = cudaMemcpy(rope, tab.data(), ntab * sizeof(float2), cudaMemcpyHostToDevice)) != cudaSuccess ||
      (e = cudaMemcpy(rank, ranks.data(), nslot * sizeof(int), cudaMemcpyHostToDevice)) != cudaSuccess)
    return give_up(e, "upload");
  cudaFree(c->rank);
  cudaFree(c->rope);
  c->rank = rank;
  c->rope = rope;
  c->rope_base = rope_base;
  c->rope_low = low;
  c->rope_hi = hi;
  // the cluster kernel with one more int of shared memory per slot; a
  // warp-per-pair or explicit shape goes back to the automatic one
  c->shape_auto = h2o::decode_pick_shape(c->dtype, c->D, c->P, c->C, entries);
  c->splits_override = 0;
  c->stages_override = 0;
  return H2O_OK;
}
}  // namespace

int h2o_cache_set_position_rolling(h2o_cache* c, float rope_base) {
  NvtxRange nvtx("h2o_cache_set_position_rolling");
  if (!c) return fail(H2O_EINVAL, "h2o_cache_set_position_rolling: cache is NULL");
  if (!(rope_base >= 0.f) || !std::isfinite(rope_base))
    return fail(H2O_EINVAL, "h2o_cache_set_position_rolling: rope_base must be finite and >= 0 (0 = off)");
  return set_rolling(c, rope_base, 0, 0, "h2o_cache_set_position_rolling");
}

int h2o_cache_set_rolling_digits(h2o_cache* c, int low_bits, int hi_bits) {
  NvtxRange nvtx("h2o_cache_set_rolling_digits");
  if (!c) return fail(H2O_EINVAL, "h2o_cache_set_rolling_digits: cache is NULL");
  if (!c->rope) return fail(H2O_ESTATE, "h2o_cache_set_rolling_digits: position rolling is off");
  const bool automatic = low_bits == 0 && hi_bits == 0;
  if (!automatic && (low_bits < h2o::kRopeMinBits || low_bits > h2o::kRopeMaxBits || hi_bits < h2o::kRopeMinBits ||
                     hi_bits > h2o::kRopeMaxBits))
    return fail(H2O_EINVAL, "h2o_cache_set_rolling_digits: digit widths must be %d..%d bits (or both 0)",
                h2o::kRopeMinBits, h2o::kRopeMaxBits);
  if (!automatic) {
    const int levels = h2o::rope_levels_for(c->C, low_bits, hi_bits);
    const h2o::DecodeShape sh =
        h2o::decode_pick_shape(c->dtype, c->D, c->P, c->C, h2o::rope_entries_for(c->C, low_bits, hi_bits));
    if (levels > 5 || h2o::decode_resident(c->dtype, c->D, sh.splits, sh.stages, chunk_for(c->C, sh.splits), c->P,
                                           h2o::rope_entries_for(c->C, low_bits, hi_bits)) < sh.splits)
      return fail(H2O_EINVAL, "h2o_cache_set_rolling_digits: %d + %d-bit digits cannot be scheduled for %d slots",
                  low_bits, hi_bits, c->C);
  }
  return set_rolling(c, c->rope_base, low_bits, hi_bits, "h2o_cache_set_rolling_digits");
}

int h2o_cache_rolling_digits(const h2o_cache* c, int32_t* digits) {
  if (!c || !digits) return fail(H2O_EINVAL, "h2o_cache_rolling_digits: NULL argument");
  digits[0] = c->rope ? c->rope_low : 0;
  digits[1] = c->rope ? c->rope_hi : 0;
  digits[2] = c->rope ? h2o::rope_levels_for(c->C, c->rope_low, c->rope_hi) : 0;
  digits[3] = c->rope ? h2o::rope_entries_for(c->C, c->rope_low, c->rope_hi) : 0;
  return H2O_OK;
}

#ifdef H2O_DECODE_TIMELINE
// Profiling build only (not declared in h2o.h): copy the decode time stamps
// [kTimelineSlots][kTimelineMaxCtas][kTimelineStamps] (uint64 ns) to host
// memory and report the buffer the next decode launch will write.
H2O_API int h2o_debug_decode_timeline(void* host_buf, size_t bytes, int* next_slot) {
  if (!host_buf || !next_slot) return fail(H2O_EINVAL, "h2o_debug_decode_timeline: NULL argument");
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = h2o::decode_timeline_read(host_buf, bytes);
  if (e != cudaSuccess) return cuda_fail(e, "h2o_debug_decode_timeline");
  *next_slot = static_cast<int>(g_tl_next.load() % h2o::kTimelineSlots);
  return H2O_OK;
}
#endif

int h2o_debug_fail_alloc(int after) {
  if (after < -1) return fail(H2O_EINVAL, "h2o_debug_fail_alloc: after must be >= -1");
  g_alloc_budget.store(after);
  return H2O_OK;
}

int h2o_selftest_wait_timeout(unsigned polls, int* gave_up, unsigned long long* elapsed_ns) {
  if (polls < 1 || polls > 1000000u || gave_up == nullptr || elapsed_ns == nullptr)
    return fail(H2O_EINVAL, "h2o_selftest_wait_timeout: polls must be 1..1000000 and the outputs non-null");
  void* buf = nullptr;
  cudaError_t e = dev_alloc(&buf, 16);
  if (e != cudaSuccess) return cuda_fail(e, "h2o_selftest_wait_timeout: cudaMalloc");
  int* flags = static_cast<int*>(buf);
  unsigned long long* ns = reinterpret_cast<unsigned long long*>(static_cast<char*>(buf) + 8);
  wait_timeout_probe<<<1, 32>>>(polls, flags, ns);
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  int host_flags[2] = {0, 0};
  unsigned long long host_ns = 0;
  if (e == cudaSuccess) e = cudaMemcpy(host_flags, flags, sizeof(host_flags), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(&host_ns, ns, sizeof(host_ns), cudaMemcpyDeviceToHost);
  cudaFree(buf);
  if (e != cudaSuccess) return cuda_fail(e, "h2o_selftest_wait_timeout");
  gave_up[0] = host_flags[0];
  gave_up[1] = host_flags[1];
  *elapsed_ns = host_ns;
  return H2O_OK;
}

}  // extern "C"
