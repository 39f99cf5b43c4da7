// H2O prefill, part 1: causal attention row statistics (log-sum-exp, optional
// output) and the column sums that seed every prompt token's accumulated
// attention score.
//
// Method: "H2O: Heavy-Hitter Oracle ... 深度解读报告", section 3.4 (prefill rule:
// keep heavy hitters + recent tokens of a long prompt) with the score of
// section 3.3 / section 2.3 (the attention mass a token has received):
//   colsum_j = sum_{i >= j} exp(s_ij - lse_i),  s_ij = scale * q_i . k_j.
// The column sums need each row's final normaliser, so the prompt is read
// twice: pass 1 computes lse_i row by row (online softmax, optionally the
// output O); pass 2 walks down each key's column and accumulates
// probabilities in a fixed order, so the result does not depend on
// scheduling.
//
// fp16 K/V: both passes run on the tcgen05 tensor cores (prefill_tc.cu).
// fp32 K/V: the plain FFMA kernels below (a TF32 contraction would not meet
// the 1e-5 tolerance of the score), float64 column accumulation.
#include <cuda_fp16.h>

#include "h2o_internal.cuh"
#include "ptx.cuh"

namespace h2o {
namespace {

constexpr float kNeg = -3.0e38f;
// ---------------------------------------------------------------- fp32 (FFMA) passes
// One warp per query row; lanes take 32 keys at a time.
template <int D>
__global__ void __launch_bounds__(128) stats_f32(const PrefillParams prm) {
  constexpr int PER = D / 32;
  __shared__ __align__(16) float qs[4][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int LS = prm.L, pair = blockIdx.y;
  const int i = blockIdx.x * 4 + warp;
  griddep_wait();
  const int L = pair_len(prm.lens, prm.heads, LS, pair);  // LS: row stride
  if (i >= L) return;
  const size_t base = static_cast<size_t>(pair) * LS * D;
  const float* Q = static_cast<const float*>(prm.q) + base;
  const float* K = static_cast<const float*>(prm.k) + base;
  const float* V = static_cast<const float*>(prm.v) + base;
  for (int d = lane; d < D; d += 32) qs[warp][d] = Q[static_cast<size_t>(i) * D + d];
  __syncwarp();
  float m = kNeg, l = 0.f, o[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) o[e] = 0.f;
  for (int kb = 0; kb <= i; kb += 32) {
    const int j = kb + lane;
    float s = -INFINITY;
    if (j <= i) {
      const float4* kr = reinterpret_cast<const float4*>(K + static_cast<size_t>(j) * D);
      float acc = 0.f;
#pragma unroll 4
      for (int d4 = 0; d4 < D / 4; ++d4) {
        const float4 kv = kr[d4];
        acc = fmaf(qs[warp][4 * d4], kv.x, acc);
        acc = fmaf(qs[warp][4 * d4 + 1], kv.y, acc);
        acc = fmaf(qs[warp][4 * d4 + 2], kv.z, acc);
        acc = fmaf(qs[warp][4 * d4 + 3], kv.w, acc);
      }
      s = acc * prm.qscale;
    }
    float mx = s;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float mn = fmaxf(m, mx);
    const float corr = exp2f(m - mn);
    m = mn;
    const float pr = exp2f(s - m);
    l = l * corr + pr;
#pragma unroll
    for (int e = 0; e < PER; ++e) o[e] *= corr;
    if (prm.out) {
      const int nk = min(32, i + 1 - kb);
      for (int jj = 0; jj < nk; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, pr, jj);
        const float* vr = V + static_cast<size_t>(kb + jj) * D;
#pragma unroll
        for (int e = 0; e < PER; ++e) o[e] = fmaf(pj, vr[lane + 32 * e], o[e]);
      }
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  if (lane == 0) prm.lse2[static_cast<size_t>(pair) * LS + i] = m + log2f(l);
  if (prm.out) {
    const float inv = 1.f / l;
#pragma unroll
    for (int e = 0; e < PER; ++e) prm.out[(static_cast<size_t>(pair) * LS + i) * D + lane + 32 * e] = o[e] * inv;
  }
}

// One warp per key column; lanes take 32 query rows at a time; float64 sum.
template <int D>
__global__ void __launch_bounds__(128) colsum_f32(const PrefillParams prm) {
  __shared__ __align__(16) float ks[4][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int LS = prm.L, pair = blockIdx.y;
  const int j = blockIdx.x * 4 + warp;
  griddep_wait();
  const int L = pair_len(prm.lens, prm.heads, LS, pair);  // LS: row stride
  if (j >= L) return;
  const size_t base = static_cast<size_t>(pair) * LS * D;
  const float* Q = static_cast<const float*>(prm.q) + base;
  const float* K = static_cast<const float*>(prm.k) + base;
  const float* lse2 = prm.lse2 + static_cast<size_t>(pair) * LS;
  for (int d = lane; d < D; d += 32) ks[warp][d] = K[static_cast<size_t>(j) * D + d];
  __syncwarp();
  double acc = 0.0;
  for (int i = j + lane; i < L; i += 32) {
    const float4* qr = reinterpret_cast<const float4*>(Q + static_cast<size_t>(i) * D);
    float dot = 0.f;
#pragma unroll 4
    for (int d4 = 0; d4 < D / 4; ++d4) {
      const float4 qv = qr[d4];
      dot = fmaf(qv.x, ks[warp][4 * d4], dot);
      dot = fmaf(qv.y, ks[warp][4 * d4 + 1], dot);
      dot = fmaf(qv.z, ks[warp][4 * d4 + 2], dot);
      dot = fmaf(qv.w, ks[warp][4 * d4 + 3], dot);
    }
    acc += static_cast<double>(exp2f(dot * prm.qscale - lse2[i]));
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) prm.colsum[static_cast<size_t>(pair) * LS + j] = static_cast<float>(acc);
}

__global__ void lse_export_kernel(const float* lse2, float* lse, size_t n) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    lse[i] = lse2[i] * 0.69314718055994530942f;
}

template <typename K>
cudaError_t launch_pdl(K kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s, const PrefillParams& prm) {
  cudaError_t e = kernel_attrs(reinterpret_cast<const void*>(kern), smem, false);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, prm);
}

}  // namespace

cudaError_t launch_prefill_stats(const PrefillParams& prm, int dtype, int D, int pairs, cudaStream_t s) {
  if (prm.L <= 0) return cudaSuccess;
  if (dtype == 0) return launch_prefill_stats_tc(prm, D, pairs, s);
  const dim3 grid((prm.L + 3) / 4, pairs);
  if (D == 128) return launch_pdl(stats_f32<128>, grid, 128, 0, s, prm);
  if (D == 64) return launch_pdl(stats_f32<64>, grid, 128, 0, s, prm);
  return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_colsum(const PrefillParams& prm, int dtype, int D, int pairs, cudaStream_t s) {
  if (prm.L <= 0) return cudaSuccess;
  if (dtype == 0)  // with the output, the output pass left partials to reduce
    return prm.out && prm.cs_part ? launch_colsum_reduce(prm, pairs, s) : launch_prefill_colsum_tc(prm, D, pairs, s);
  const dim3 grid((prm.L + 3) / 4, pairs);
  if (D == 128) return launch_pdl(colsum_f32<128>, grid, 128, 0, s, prm);
  if (D == 64) return launch_pdl(colsum_f32<64>, grid, 128, 0, s, prm);
  return cudaErrorInvalidValue;
}

cudaError_t launch_lse_export(const float* lse2, float* lse, size_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int blocks = static_cast<int>(n < 256 * 1024 ? (n + 255) / 256 : 1024);
  lse_export_kernel<<<blocks, 256, 0, s>>>(lse2, lse, n);
  return cudaGetLastError();
}

}  // namespace h2o
