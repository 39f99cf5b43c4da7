// Prefill column sums for callers that cannot allocate device memory.
//
// Some host programs own every byte of device memory themselves: engines that
// carve all GPU memory into their own pools at start-up and forbid any later
// cudaMalloc, or latency-bound loops where cudaMalloc's implicit device-wide
// synchronisation is not acceptable.  h2o_prefill_colsum_static serves them:
// it runs the same two prefill kernels as h2o_prefill_ex (row log-sum-exp,
// then column sums) but keeps the row statistics, its only scratch, in a
// fixed array in the library's own device memory instead of a workspace it
// would have to allocate.
#include <cuda_runtime.h>

#include <mutex>

#include "h2o.h"
#include "h2o_internal.cuh"

namespace {

// 2^21 floats = 8 MiB: B*H*L up to 2,097,152 (e.g. 32 heads x 16384 tokens,
// or 256 pairs x 8192 tokens).  Every GPU that loads the library holds this
// array until the process exits.
constexpr size_t kScratchFloats = size_t(1) << 21;
static __device__ __align__(256) float g_colsum_scratch[kScratchFloats];
// Device error bits of the last call's kernels (a bounded wait that gave up
// leaves some row statistics unwritten, so that call's column sums are not
// valid).  Cleared at the start of every call, read by
// h2o_prefill_colsum_static_check.
static __device__ __align__(16) int g_colsum_static_err;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};
int* g_err_ptr[kMaxDevices] = {};

// Device addresses of the scratch array and the error word on the current
// device.  The host-side symbols are only stand-ins, so the addresses are
// looked up once per device (with that device current) and cached.
int symbols_for_current_device(const char* who, float** scratch, int** err) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return h2o::set_error(H2O_ECUDA, "%s: cudaGetDevice: %s", who, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return h2o::set_error(H2O_EINVAL, "%s: device %d unsupported", who, dev);
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev] || !g_err_ptr[dev]) {
    void* p = nullptr;
    void* q = nullptr;
    e = cudaGetSymbolAddress(&p, g_colsum_scratch);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(&q, g_colsum_static_err);
    if (e != cudaSuccess || !p || !q)
      return h2o::set_error(H2O_ECUDA, "%s: cudaGetSymbolAddress: %s", who, cudaGetErrorString(e));
    g_scratch_ptr[dev] = static_cast<float*>(p);
    g_err_ptr[dev] = static_cast<int*>(q);
  }
  if (scratch) *scratch = g_scratch_ptr[dev];
  if (err) *err = g_err_ptr[dev];
  return H2O_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" H2O_API int h2o_prefill_colsum_static(const void* q, const void* k, int batch, int heads, int head_dim,
                                                 int prompt_len, int kv_dtype, float scale, float* colsum,
                                                 void* stream) {
  if (!q || !k || !colsum) return h2o::set_error(H2O_EINVAL, "h2o_prefill_colsum_static: q, k and colsum are required");
  if (batch < 1 || heads < 1 || prompt_len < 1)
    return h2o::set_error(H2O_EINVAL, "h2o_prefill_colsum_static: batch, heads and prompt_len must be >= 1");
  if (head_dim != 64 && head_dim != 128)
    return h2o::set_error(H2O_EINVAL, "h2o_prefill_colsum_static: head_dim must be 64 or 128");
  if (kv_dtype != H2O_F16 && kv_dtype != H2O_F32)
    return h2o::set_error(H2O_EINVAL, "h2o_prefill_colsum_static: bad kv_dtype");
  if (!(scale > 0.f)) return h2o::set_error(H2O_EINVAL, "h2o_prefill_colsum_static: scale must be positive");
  if (!aligned16(q) || !aligned16(k))
    return h2o::set_error(H2O_EINVAL, "h2o_prefill_colsum_static: q and k must be 16-byte aligned");
  const long long pairs = static_cast<long long>(batch) * heads;
  const long long need = pairs * prompt_len;
  if (pairs > 65535 || need > static_cast<long long>(kScratchFloats))
    return h2o::set_error(H2O_EINVAL,
                "h2o_prefill_colsum_static: batch*heads*prompt_len = %lld exceeds the fixed scratch of %zu floats",
                need, kScratchFloats);
  float* scratch = nullptr;
  int* err = nullptr;
  int rc = symbols_for_current_device("h2o_prefill_colsum_static", &scratch, &err);
  if (rc != H2O_OK) return rc;
  // Every entry of the scratch that the column-sum pass reads is written by
  // the row-statistics pass of this call first, so the scratch is not
  // cleared; only the error word must start at zero.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(err, 0, sizeof(int), s);
  if (e != cudaSuccess)
    return h2o::set_error(H2O_ECUDA, "h2o_prefill_colsum_static: clear error word: %s", cudaGetErrorString(e));
  h2o::PrefillParams pp;
  pp.q = q;
  pp.k = k;
  pp.v = nullptr;  // no attention output: V is not read
  pp.out = nullptr;
  pp.lse2 = scratch;
  pp.colsum = colsum;
  pp.L = prompt_len;
  pp.qscale = scale * 1.4426950408889634f;
  pp.err = err;
  e = h2o::launch_prefill_stats(pp, kv_dtype, head_dim, static_cast<int>(pairs), s);
  if (e == cudaSuccess) e = h2o::launch_prefill_colsum(pp, kv_dtype, head_dim, static_cast<int>(pairs), s);
  if (e != cudaSuccess)
    return h2o::set_error(H2O_ECUDA, "h2o_prefill_colsum_static: launch: %s", cudaGetErrorString(e));
  return H2O_OK;
}

extern "C" H2O_API int h2o_prefill_colsum_static_check(void* stream) {
  int* err = nullptr;
  int rc = symbols_for_current_device("h2o_prefill_colsum_static_check", nullptr, &err);
  if (rc != H2O_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int flags = 0;
  cudaError_t e = cudaMemcpyAsync(&flags, err, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess)
    return h2o::set_error(H2O_ECUDA, "h2o_prefill_colsum_static_check: %s", cudaGetErrorString(e));
  if (flags)
    return h2o::set_error(H2O_EDEVICE,
                          "h2o_prefill_colsum_static_check: a bounded wait gave up (flags 0x%x); the last call's "
                          "column sums are not valid", flags);
  return H2O_OK;
}
