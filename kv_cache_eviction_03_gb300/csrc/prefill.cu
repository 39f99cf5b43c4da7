// H2O prefill, part 1: causal attention row statistics (log-sum-exp, optional
// output) and the column sums that seed every prompt token's accumulated
// attention score.
//
// Method: "H2O: Heavy-Hitter Oracle ... 深度解读报告", section 3.4 (prefill rule:
// keep heavy hitters + recent tokens of a long prompt) with the score of
// section 3.3 / section 2.3 (the attention mass a token has received):
//   colsum_j = sum_{i >= j} exp(s_ij - lse_i),  s_ij = scale * q_i . k_j.
// The column sums need each row's final normaliser, so the prompt is read
// twice: pass 1 (stats_*) computes lse_i row by row (flash-attention style
// online softmax, optionally the output O); pass 2 (colsum_*) walks down each
// key block's column and accumulates probabilities in a fixed order (float32
// within a 64-row query block, float64 across blocks), so the result does not
// depend on scheduling.
//
// fp16 K/V: the q.k and p.v contractions run on tensor cores (mma.sync
// m16n8k16, fp32 accumulators, ldmatrix from XOR-swizzled shared memory,
// cp.async double buffering).  fp32 K/V: plain FFMA (a TF32 contraction would
// not meet the 1e-5 tolerance of the score).
#include <cuda_fp16.h>

#include <cstdlib>
#include <cstring>

#include "h2o_internal.cuh"
#include "ptx.cuh"

namespace h2o {
namespace {

constexpr float kNeg = -3.0e38f;
constexpr int BM = 64;  // query rows per CTA (stats) / per query block (colsum)
constexpr int BN = 64;  // keys per key block

// byte offset of 16-byte chunk `ch` of row `r` in a [rows][D] fp16 tile whose
// chunks are XOR-swizzled by the row index (conflict-free ldmatrix)
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int ch) {
  return static_cast<uint32_t>(r * D * 2 + ((ch ^ (r & 7)) << 4));
}

// Copy `BM` rows (row0..) of a [L, D] fp16 matrix into a swizzled tile;
// rows >= L are zero-filled.
template <int D, int NT>
__device__ __forceinline__ void load_tile(unsigned char* tile, const __half* src, int row0, int L, int tid) {
  constexpr int CH = D / 8;
  for (int c = tid; c < BM * CH; c += NT) {
    const int r = c / CH, ch = c % CH;
    const int gr = row0 + r;
    const bool ok = gr < L;
    cp_async16(tile + swz<D>(r, ch), src + static_cast<size_t>(ok ? gr : 0) * D + ch * 8, ok);
  }
}

// ---------------------------------------------------------------- pass 1, fp16
template <int D, bool WITH_O>
__global__ void __launch_bounds__(128) stats_f16(const PrefillParams prm) {
  constexpr int KS = D / 16;  // k16 steps over the head dimension
  constexpr int DT = D / 8;   // n8 tiles over the head dimension
  constexpr int TILE = BM * D * 2;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* sQ = smem;
  unsigned char* sK = smem + TILE;                 // [2] tiles
  unsigned char* sV = smem + 3 * TILE;             // [2] tiles (WITH_O)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int LS = prm.L;  // row stride; L below is this pair's prompt length
  const int pair = blockIdx.y;
  const int qb = gridDim.x - 1 - blockIdx.x;  // longest rows first
  const int q0 = qb * BM;
  const size_t base = static_cast<size_t>(pair) * LS * D;
  const __half* Q = static_cast<const __half*>(prm.q) + base;
  const __half* K = static_cast<const __half*>(prm.k) + base;
  const __half* V = static_cast<const __half*>(prm.v) + base;

  griddep_wait();
  const int L = pair_len(prm.lens, prm.heads, LS, pair);
  if (q0 >= L) return;
  load_tile<D, 128>(sQ, Q, q0, L, tid);
  load_tile<D, 128>(sK, K, 0, L, tid);
  if (WITH_O) load_tile<D, 128>(sV, V, 0, L, tid);
  cp_async_commit();

  uint32_t qf[KS][4];
  float m[2] = {kNeg, kNeg}, l[2] = {0.f, 0.f};
  float o[WITH_O ? DT : 1][4];
#pragma unroll
  for (int i = 0; i < (WITH_O ? DT : 1); ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  const int row_g = q0 + warp * 16 + g;  // this thread's rows: row_g, row_g + 8

  const int nkb = qb + 1;
  for (int kb = 0; kb < nkb; ++kb) {
    const int buf = kb & 1;
    if (kb + 1 < nkb) {
      load_tile<D, 128>(sK + (buf ^ 1) * TILE, K, (kb + 1) * BN, L, tid);
      if (WITH_O) load_tile<D, 128>(sV + (buf ^ 1) * TILE, V, (kb + 1) * BN, L, tid);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (kb == 0) {
      const uint32_t qa = smem_u32(sQ);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
        ldsm_x4(qa + swz<D>(warp * 16 + (lane & 15), 2 * ks + (lane >> 4)), qf[ks][0], qf[ks][1], qf[ks][2],
                qf[ks][3]);
    }
    // S = Q K^T for 16 rows x 64 keys
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    const uint32_t ka = smem_u32(sK + buf * TILE);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(ka + swz<D>(np * 16 + (lane & 7) + ((lane >> 4) << 3), 2 * ks + ((lane >> 3) & 1)), b0, b1, b2,
                b3);
        mma_f16_16816(s[2 * np], qf[ks], b0, b1);
        mma_f16_16816(s[2 * np + 1], qf[ks], b2, b3);
      }
    }
    // scale into the base-2 domain, causal / length mask, online softmax
    float mx[2] = {kNeg, kNeg};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int kj = kb * BN + nt * 8 + 2 * t4 + (c & 1);
        const int qi = row_g + ((c >> 1) << 3);
        const float x = (kj <= qi && kj < L) ? s[nt][c] * prm.qscale : -INFINITY;
        s[nt][c] = x;
        mx[c >> 1] = fmaxf(mx[c >> 1], x);
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
    }
    float corr[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float mn = fmaxf(m[h], mx[h]);
      corr[h] = exp2f(m[h] - mn);
      m[h] = mn;
      l[h] *= corr[h];
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float pr = exp2f(s[nt][c] - m[c >> 1]);
        s[nt][c] = pr;
        l[c >> 1] += pr;
      }
    }
    if (WITH_O) {
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) {
        o[dt][0] *= corr[0];
        o[dt][1] *= corr[0];
        o[dt][2] *= corr[1];
        o[dt][3] *= corr[1];
      }
      const uint32_t va = smem_u32(sV + buf * TILE);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t a[4];
        a[0] = pack_half2(s[2 * kk][0], s[2 * kk][1]);
        a[1] = pack_half2(s[2 * kk][2], s[2 * kk][3]);
        a[2] = pack_half2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        a[3] = pack_half2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
        for (int dp = 0; dp < DT / 2; ++dp) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(va + swz<D>(kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3), 2 * dp + (lane >> 4)), b0, b1,
                    b2, b3);
          mma_f16_16816(o[2 * dp], a, b0, b1);
          mma_f16_16816(o[2 * dp + 1], a, b2, b3);
        }
      }
    }
    __syncthreads();  // buffer `buf` is refilled next iteration
  }
  griddep_launch();
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int qi = row_g + h * 8;
    if (qi < L) {
      if (t4 == 0) prm.lse2[static_cast<size_t>(pair) * LS + qi] = m[h] + log2f(l[h]);
      if (WITH_O) {
        const float inv = 1.f / l[h];
        float* orow = prm.out + (static_cast<size_t>(pair) * LS + qi) * D;
#pragma unroll
        for (int dt = 0; dt < DT; ++dt)
          *reinterpret_cast<float2*>(orow + dt * 8 + 2 * t4) =
              make_float2(o[dt][2 * h] * inv, o[dt][2 * h + 1] * inv);
      }
    }
  }
}

// ---------------------------------------------------------------- pass 2, fp16
template <int D>
__global__ void __launch_bounds__(128) colsum_f16(const PrefillParams prm) {
  constexpr int KS = D / 16;
  constexpr int TILE = BM * D * 2;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* sK = smem;
  unsigned char* sQ = smem + TILE;                                  // [2] tiles
  float* sL = reinterpret_cast<float*>(smem + 3 * TILE);            // [2][BM] lse2
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int LS = prm.L;  // row stride; L below is this pair's prompt length
  const int pair = blockIdx.y;
  const int jb = blockIdx.x;  // key block; block 0 has the most query blocks
  const size_t base = static_cast<size_t>(pair) * LS * D;
  const __half* Q = static_cast<const __half*>(prm.q) + base;
  const __half* K = static_cast<const __half*>(prm.k) + base;
  const float* lse2 = prm.lse2 + static_cast<size_t>(pair) * LS;
  

  griddep_wait();
  const int L = pair_len(prm.lens, prm.heads, LS, pair);
  const int nqb = (L + BM - 1) / BM;
  if (jb * BN >= L) return;
  load_tile<D, 128>(sK, K, jb * BN, L, tid);
  load_tile<D, 128>(sQ, Q, jb * BM, L, tid);
  for (int r = tid; r < BM; r += 128) {
    const int qi = jb * BM + r;
    sL[r] = qi < L ? lse2[qi] : 0.f;
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();

  uint32_t kf[KS][4];  // this warp's 16 keys: [ks][b0,b1 of n-tile 0, b0,b1 of n-tile 1]
  {
    const uint32_t ka = smem_u32(sK);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
      ldsm_x4(ka + swz<D>(warp * 16 + (lane & 7) + ((lane >> 4) << 3), 2 * ks + ((lane >> 3) & 1)), kf[ks][0],
              kf[ks][1], kf[ks][2], kf[ks][3]);
  }
  double acc[2][2] = {{0.0, 0.0}, {0.0, 0.0}};
  const int key0 = jb * BN + warp * 16;

  for (int qb = jb; qb < nqb; ++qb) {
    const int buf = (qb - jb) & 1;
    if (qb + 1 < nqb) {
      load_tile<D, 128>(sQ + (buf ^ 1) * TILE, Q, (qb + 1) * BM, L, tid);
      cp_async_commit();
      for (int r = tid; r < BM; r += 128) {
        const int qi = (qb + 1) * BM + r;
        sL[(buf ^ 1) * BM + r] = qi < L ? lse2[qi] : 0.f;
      }
    }
    const uint32_t qa = smem_u32(sQ + buf * TILE);
    float cs[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
    for (int mt = 0; mt < BM / 16; ++mt) {
      float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t a[4];
        ldsm_x4(qa + swz<D>(mt * 16 + (lane & 15), 2 * ks + (lane >> 4)), a[0], a[1], a[2], a[3]);
        mma_f16_16816(s[0], a, kf[ks][0], kf[ks][1]);
        mma_f16_16816(s[1], a, kf[ks][2], kf[ks][3]);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = mt * 16 + g + h * 8;
        const int qi = qb * BM + r;
        const float ls = sL[buf * BM + r];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int kj = key0 + nt * 8 + 2 * t4 + c;
            const float pr = (kj <= qi && qi < L) ? exp2f(fmaf(s[nt][2 * h + c], prm.qscale, -ls)) : 0.f;
            cs[nt][c] += pr;
          }
        }
      }
    }
    // sum the 8 row groups of the warp; lanes 0..3 then hold 64-row column sums
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float v = cs[nt][c];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        acc[nt][c] += static_cast<double>(v);
      }
    }
    if (qb + 1 < nqb) cp_async_wait<0>();
    __syncthreads();
  }
  griddep_launch();
  if (g == 0) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int kj = key0 + nt * 8 + 2 * t4 + c;
        if (kj < L) prm.colsum[static_cast<size_t>(pair) * LS + kj] = static_cast<float>(acc[nt][c]);
      }
    }
  }
}

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

// fp16 prefill engine: the tcgen05 kernels unless H2O_PREFILL_ENGINE=mma
// selects the mma.sync ones (kept for comparison).
bool prefill_use_tc() {
  static const bool tc = [] {
    const char* v = std::getenv("H2O_PREFILL_ENGINE");
    return !(v && std::strcmp(v, "mma") == 0);
  }();
  return tc;
}

cudaError_t launch_prefill_stats(const PrefillParams& prm, int dtype, int D, int pairs, cudaStream_t s) {
  if (prm.L <= 0) return cudaSuccess;
  if (dtype == 0 && prefill_use_tc()) return launch_prefill_stats_tc(prm, D, pairs, s);
  if (dtype == 0) {
    const dim3 grid((prm.L + BM - 1) / BM, pairs);
    const bool wo = prm.out != nullptr;
    const size_t smem = static_cast<size_t>(BM) * D * 2 * (wo ? 5 : 3);
    if (D == 128) return wo ? launch_pdl(stats_f16<128, true>, grid, 128, smem, s, prm)
                            : launch_pdl(stats_f16<128, false>, grid, 128, smem, s, prm);
    if (D == 64) return wo ? launch_pdl(stats_f16<64, true>, grid, 128, smem, s, prm)
                           : launch_pdl(stats_f16<64, false>, grid, 128, smem, s, prm);
  } else {
    const dim3 grid((prm.L + 3) / 4, pairs);
    if (D == 128) return launch_pdl(stats_f32<128>, grid, 128, 0, s, prm);
    if (D == 64) return launch_pdl(stats_f32<64>, grid, 128, 0, s, prm);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_colsum(const PrefillParams& prm, int dtype, int D, int pairs, cudaStream_t s) {
  if (prm.L <= 0) return cudaSuccess;
  if (dtype == 0 && prefill_use_tc())  // with the output, the output pass left partials to reduce
    return prm.out && prm.cs_part ? launch_colsum_reduce(prm, pairs, s) : launch_prefill_colsum_tc(prm, D, pairs, s);
  if (dtype == 0) {
    const dim3 grid((prm.L + BN - 1) / BN, pairs);
    const size_t smem = static_cast<size_t>(BM) * D * 2 * 3 + 2 * BM * sizeof(float);
    if (D == 128) return launch_pdl(colsum_f16<128>, grid, 128, smem, s, prm);
    if (D == 64) return launch_pdl(colsum_f16<64>, grid, 128, smem, s, prm);
  } else {
    const dim3 grid((prm.L + 3) / 4, pairs);
    if (D == 128) return launch_pdl(colsum_f32<128>, grid, 128, 0, s, prm);
    if (D == 64) return launch_pdl(colsum_f32<64>, grid, 128, 0, s, prm);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_lse_export(const float* lse2, float* lse, size_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int blocks = static_cast<int>(n < 256 * 1024 ? (n + 255) / 256 : 1024);
  lse_export_kernel<<<blocks, 256, 0, s>>>(lse2, lse, n);
  return cudaGetLastError();
}

}  // namespace h2o
