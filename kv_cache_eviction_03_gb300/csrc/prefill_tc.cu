// H2O prefill on the 5th-generation tensor cores (tcgen05, accumulators in
// tensor memory): the row log-sum-exp pass and the column-sum pass for fp16
// K/V.
//
// Method: "H2O: Heavy-Hitter Oracle ... 深度解读报告", section 3.4 (prefill
// keep rule) with the score of section 3.3 / 2.3: every prompt token's score
// is the attention mass it receives, colsum_j = sum_{i>=j} exp(s_ij - lse_i),
// s_ij = scale * q_i . k_j.
//
// Both passes work on 128 x 128 blocks of logits.  One thread issues
// tcgen05.mma (M = N = 128, K = 16, fp16 operands from shared memory laid out
// K-major with the 128-byte swizzle, fp32 accumulators in TMEM); the block's
// 256 threads then read the accumulators with tcgen05.ld and do the
// exponentials.  Two TMEM accumulators and two operand stages let the tensor
// core work on block i+1 while the threads finish block i.
//  - rows (stats_tc): A = 128 query rows, B = a 128-key block; TMEM lane =
//    query row, so each thread keeps an online max / sum of its row.
//  - columns (colsum_tc): A = 128 keys, B = a 128-query block, i.e. the
//    transposed logits; TMEM lane = key, so each thread sums the
//    probabilities its key receives with no cross-thread reduction (float32
//    within a block, float64 across blocks: fixed order, deterministic).
// Every wait is bounded; the TMEM allocation is freed on every path.
#include <cuda_fp16.h>

#include "h2o_internal.cuh"
#include "ptx.cuh"

namespace h2o {
namespace {

constexpr float kNeg = -3.0e38f;
constexpr uint32_t kWaitLimit = 200000u;  // polls of <= 1 us: waits on this CTA's own MMAs
constexpr int NT = 256;                    // 8 warps: 4 TMEM lane quarters x 2 column halves
constexpr int BLK = 128;                   // rows / columns of a logits block
constexpr uint32_t kTmemCols = 256;        // two 128-column fp32 accumulators
constexpr size_t kMinSmem = 100 * 1024;    // at most two CTAs per SM: 2 x 256 TMEM columns fit

template <int D>
struct TcCfg {
  static constexpr int TILE = BLK * D * 2;                  // one operand tile (bytes)
  static constexpr int KB = BLK * 128;                      // bytes of one 64-element K block
  static constexpr size_t tiles = 3 * static_cast<size_t>(TILE);  // fixed operand + 2 stages
  static constexpr size_t lse = tiles;                      // [3][128] floats
  static constexpr size_t bars = lse + 3 * BLK * 4;         // 2 mbarriers
  static constexpr size_t tslot = bars + 16;                // TMEM base address
  static constexpr size_t red = (tslot + 16 + 15) / 16 * 16;  // [128] doubles / float pairs
  static constexpr size_t used = red + BLK * 8 * 2;
  // + 1 KB so the operand tiles can start on a 1024-byte boundary
  static constexpr size_t bytes = (used > kMinSmem ? used : kMinSmem) + 1024;
};

// 128 rows (row0..) of a [L, D] fp16 matrix into a K-major 128-byte-swizzled
// tile: 64-element K block kb at tile + kb * 16 KB, row r at + r * 128 B,
// 16-byte chunk c at chunk c ^ (r % 8).  Rows >= L are zero-filled.
template <int D>
__device__ __forceinline__ void load_tile(unsigned char* tile, const __half* src, int row0, int L, int tid) {
  constexpr int CPR = D / 8;  // 16-byte chunks per row
  for (int c = tid; c < BLK * CPR; c += NT) {
    const int r = c / CPR, ch = c % CPR;
    const int gr = row0 + r;
    const bool ok = gr < L;
    unsigned char* dst = tile + (ch >> 3) * TcCfg<D>::KB + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
    cp_async16(dst, src + static_cast<size_t>(ok ? gr : 0) * D + ch * 8, ok);
  }
}

// Log2-domain lse of query row row0 + t; rows past the prompt get a huge
// value so that their probabilities exp2(s - lse) vanish without a mask.  A
// plain load: the rows of the vector need not be 16-byte aligned.
constexpr float kHugeLse = 3.0e38f;
__device__ __forceinline__ float lse_at(const float* src, int row0, int t, int L) {
  return row0 + t < L ? src[row0 + t] : kHugeLse;
}

// D[tmem] = A[128 x D] * B[128 x D]^T over the head dimension.
template <int D>
__device__ __forceinline__ void issue_block(uint32_t d_tmem, const unsigned char* a, const unsigned char* b) {
  constexpr uint32_t idesc = tc::idesc_f16_f32(BLK, BLK);
  const uint32_t sa = smem_u32(a), sb = smem_u32(b);
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const uint32_t off = static_cast<uint32_t>((ks >> 2) * TcCfg<D>::KB + (ks & 3) * 32);
    tc::mma_f16(d_tmem, tc::desc_k_sw128(sa + off), tc::desc_k_sw128(sb + off), idesc, ks > 0);
  }
}

// ---------------------------------------------------------------- column sums
// The 128-byte swizzle is a function of address bits 4..9, so the operand
// tiles start on a 1024-byte boundary of the shared window.
__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
  return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
}

template <int D>
__global__ void __launch_bounds__(NT, 2) colsum_tc(const PrefillParams prm) {
  using Cfg = TcCfg<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  unsigned char* sK = smem;
  unsigned char* sQ0 = smem + Cfg::TILE;
  float* sL = reinterpret_cast<float*>(smem + Cfg::lse);
  uint64_t* mb = reinterpret_cast<uint64_t*>(smem + Cfg::bars);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + Cfg::tslot);
  double* red = reinterpret_cast<double*>(smem + Cfg::red);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = prm.L, pair = blockIdx.y, kb = blockIdx.x;
  const size_t base = static_cast<size_t>(pair) * L * D;
  const __half* Q = static_cast<const __half*>(prm.q) + base;
  const __half* K = static_cast<const __half*>(prm.k) + base;
  const float* lse2 = prm.lse2 + static_cast<size_t>(pair) * L;
  const int n = (L + BLK - 1) / BLK - kb;  // query blocks from the diagonal down

  griddep_wait();
  if (warp == 0) tc::tmem_alloc(tslot, kTmemCols);
  if (tid == 0) {
    mbar_init(&mb[0], 1);
    mbar_init(&mb[1], 1);
    fence_mbar_init();
  }
  load_tile<D>(sK, K, kb * BLK, L, tid);
  load_tile<D>(sQ0, Q, kb * BLK, L, tid);
  if (n > 1) load_tile<D>(sQ0 + Cfg::TILE, Q, (kb + 1) * BLK, L, tid);
  if (tid < BLK) {
    sL[tid] = lse_at(lse2, kb * BLK, tid, L);
    sL[BLK + tid] = lse_at(lse2, (kb + 1) * BLK, tid, L);
  }
  cp_async_commit();
  cp_async_wait<0>();
  fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tslot;
  if (tid == 0) {
    issue_block<D>(tbase, sK, sQ0);
    tc::mma_commit(&mb[0]);
    if (n > 1) {
      issue_block<D>(tbase + BLK, sK, sQ0 + Cfg::TILE);
      tc::mma_commit(&mb[1]);
    }
  }
  const int quarter = warp & 3, half = warp >> 2;
  const int key = kb * BLK + quarter * 32 + lane;  // this thread's TMEM lane
  const uint32_t lane_addr = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
  double dacc = 0.0;
  bool ok = true;
  int waited = 0;  // MMAs known complete
  for (int i = 0; i < n; ++i) {
    const int b = i & 1, qb = kb + i;  // query block of this iteration
    if (ok) {  // warp-uniform, so the .sync.aligned TMEM loads below never diverge
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&mb[b], static_cast<uint32_t>((i >> 1) & 1), kWaitLimit));
      if (!ok && lane == 0 && prm.err) atomicOr(prm.err, ERR_MMA_TIMEOUT);
    }
    if (ok) waited = i + 1;
    tc::fence_after_sync();
    // the tensor core is done with stage b: bring in query block i + 2
    // (its lse row is loaded now and stored after the exponentials)
    float next_lse = kHugeLse;
    if (i + 2 < n) {
      load_tile<D>(sQ0 + b * Cfg::TILE, Q, (qb + 2) * BLK, L, tid);
      if (tid < BLK) next_lse = lse_at(lse2, (qb + 2) * BLK, tid, L);
    }
    cp_async_commit();
    float acc0 = 0.f, acc1 = 0.f;
    const float* lse = sL + (i % 3) * BLK;
    if (ok) {
      const int kl = quarter * 32 + lane;  // key within the block
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float v[32];
        const int col0 = half * 64 + c * 32;
        tc::tmem_ld32(lane_addr + static_cast<uint32_t>(b * BLK + col0), v);
        const float4* l4 = reinterpret_cast<const float4*>(lse + col0);
        if (i == 0) {  // diagonal block: query col0 + e sees key kl only if kl <= col0 + e
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 t = l4[j];
            const int e = 4 * j;
            acc0 += kl <= col0 + e ? ex2(fmaf(v[e], prm.qscale, -t.x)) : 0.f;
            acc1 += kl <= col0 + e + 1 ? ex2(fmaf(v[e + 1], prm.qscale, -t.y)) : 0.f;
            acc0 += kl <= col0 + e + 2 ? ex2(fmaf(v[e + 2], prm.qscale, -t.z)) : 0.f;
            acc1 += kl <= col0 + e + 3 ? ex2(fmaf(v[e + 3], prm.qscale, -t.w)) : 0.f;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 t = l4[j];
            const int e = 4 * j;
            acc0 += ex2(fmaf(v[e], prm.qscale, -t.x));
            acc1 += ex2(fmaf(v[e + 1], prm.qscale, -t.y));
            acc0 += ex2(fmaf(v[e + 2], prm.qscale, -t.z));
            acc1 += ex2(fmaf(v[e + 3], prm.qscale, -t.w));
          }
        }
      }
    }
    const float acc = acc0 + acc1;
    dacc += static_cast<double>(acc);
    if (i + 2 < n && tid < BLK) sL[((i + 2) % 3) * BLK + tid] = next_lse;
    tc::fence_before_sync();
    cp_async_wait<0>();
    fence_proxy_async_smem();
    __syncthreads();  // accumulator b is read; query block i + 2 is in stage b
    tc::fence_after_sync();
    if (tid == 0 && ok && i + 2 < n) {
      issue_block<D>(tbase + b * BLK, sK, sQ0 + b * Cfg::TILE);
      tc::mma_commit(&mb[b]);
    }
  }
  griddep_launch();
  // after a timed-out wait, give the MMAs still in flight a bounded chance to
  // finish before the accumulators are freed
  if (tid == 0 && !ok) {
    const int issued = n < 2 ? n : min(n, waited + 2);
    for (int i = waited; i < issued; ++i) mbar_wait_bounded(&mb[i & 1], static_cast<uint32_t>((i >> 1) & 1), kWaitLimit);
  }
  if (half == 1) red[quarter * 32 + lane] = dacc;
  tc::fence_before_sync();
  __syncthreads();
  if (half == 0 && key < L)
    prm.colsum[static_cast<size_t>(pair) * L + key] = static_cast<float>(dacc + red[quarter * 32 + lane]);
  __syncwarp();
  if (warp == 0) tc::tmem_free(tbase, kTmemCols);
}

// ------------------------------------------------------- row log-sum-exp only
template <int D>
__global__ void __launch_bounds__(NT, 2) stats_tc(const PrefillParams prm) {
  using Cfg = TcCfg<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  unsigned char* sQ = smem;
  unsigned char* sK0 = smem + Cfg::TILE;
  uint64_t* mb = reinterpret_cast<uint64_t*>(smem + Cfg::bars);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + Cfg::tslot);
  float* red = reinterpret_cast<float*>(smem + Cfg::red);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = prm.L, pair = blockIdx.y;
  const int qb = gridDim.x - 1 - blockIdx.x;  // longest rows first
  const size_t base = static_cast<size_t>(pair) * L * D;
  const __half* Q = static_cast<const __half*>(prm.q) + base;
  const __half* K = static_cast<const __half*>(prm.k) + base;
  const int n = qb + 1;  // key blocks 0..qb (causal)

  griddep_wait();
  if (warp == 0) tc::tmem_alloc(tslot, kTmemCols);
  if (tid == 0) {
    mbar_init(&mb[0], 1);
    mbar_init(&mb[1], 1);
    fence_mbar_init();
  }
  load_tile<D>(sQ, Q, qb * BLK, L, tid);
  load_tile<D>(sK0, K, 0, L, tid);
  if (n > 1) load_tile<D>(sK0 + Cfg::TILE, K, BLK, L, tid);
  cp_async_commit();
  cp_async_wait<0>();
  fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tslot;
  if (tid == 0) {
    issue_block<D>(tbase, sQ, sK0);
    tc::mma_commit(&mb[0]);
    if (n > 1) {
      issue_block<D>(tbase + BLK, sQ, sK0 + Cfg::TILE);
      tc::mma_commit(&mb[1]);
    }
  }
  const int quarter = warp & 3, half = warp >> 2;
  const int row = qb * BLK + quarter * 32 + lane;  // this thread's query row (TMEM lane)
  const uint32_t lane_addr = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
  float m = kNeg, l = 0.f;
  bool ok = true;
  int waited = 0;
  for (int i = 0; i < n; ++i) {
    const int b = i & 1;
    if (ok) {  // warp-uniform, so the .sync.aligned TMEM loads below never diverge
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&mb[b], static_cast<uint32_t>((i >> 1) & 1), kWaitLimit));
      if (!ok && lane == 0 && prm.err) atomicOr(prm.err, ERR_MMA_TIMEOUT);
    }
    if (ok) waited = i + 1;
    tc::fence_after_sync();
    if (i + 2 < n) load_tile<D>(sK0 + b * Cfg::TILE, K, (i + 2) * BLK, L, tid);
    cp_async_commit();
    if (ok) {
      float v[64];
      tc::tmem_ld32(lane_addr + static_cast<uint32_t>(b * BLK + half * 64), *reinterpret_cast<float(*)[32]>(v));
      tc::tmem_ld32(lane_addr + static_cast<uint32_t>(b * BLK + half * 64 + 32),
                    *reinterpret_cast<float(*)[32]>(v + 32));
      if (i == qb) {  // diagonal block: key half * 64 + e is visible to row rl if it is <= rl
        const int rl = quarter * 32 + lane;
#pragma unroll
        for (int e = 0; e < 64; ++e) v[e] = half * 64 + e <= rl ? v[e] : -INFINITY;
      }
      // the max of the raw logits (scale > 0 commutes with max)
      float c0 = v[0], c1 = v[1];
#pragma unroll
      for (int e = 2; e < 64; e += 2) {
        c0 = fmaxf(c0, v[e]);
        c1 = fmaxf(c1, v[e + 1]);
      }
      const float mn = fmaxf(m, fmaxf(c0, c1) * prm.qscale);
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int e = 0; e < 64; e += 2) {
        s0 += ex2(fmaf(v[e], prm.qscale, -mn));
        s1 += ex2(fmaf(v[e + 1], prm.qscale, -mn));
      }
      l = l * ex2(m - mn) + (s0 + s1);
      m = mn;
    }
    tc::fence_before_sync();
    cp_async_wait<0>();
    fence_proxy_async_smem();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0 && ok && i + 2 < n) {
      issue_block<D>(tbase + b * BLK, sQ, sK0 + b * Cfg::TILE);
      tc::mma_commit(&mb[b]);
    }
  }
  griddep_launch();
  if (tid == 0 && !ok) {
    const int issued = n < 2 ? n : min(n, waited + 2);
    for (int i = waited; i < issued; ++i) mbar_wait_bounded(&mb[i & 1], static_cast<uint32_t>((i >> 1) & 1), kWaitLimit);
  }
  if (half == 1) {
    red[2 * (quarter * 32 + lane)] = m;
    red[2 * (quarter * 32 + lane) + 1] = l;
  }
  tc::fence_before_sync();
  __syncthreads();
  if (half == 0 && row < L) {
    const float m2 = red[2 * (quarter * 32 + lane)], l2 = red[2 * (quarter * 32 + lane) + 1];
    const float M = fmaxf(m, m2);
    prm.lse2[static_cast<size_t>(pair) * L + row] = M + log2f(l * ex2(m - M) + l2 * ex2(m2 - M));
  }
  __syncwarp();
  if (warp == 0) tc::tmem_free(tbase, kTmemCols);
}

// ------------------------------------------------------- attention output O
// With every row's lse known, O_i = sum_j exp2(s_ij - lse_i) v_j needs no
// online rescaling: per key block, S = Q K^T goes to TMEM, the threads turn
// it into fp16 probabilities in a K-major shared tile, and O += P V
// accumulates in TMEM across all key blocks (V as stored, [key][d], is the
// MN-major B operand: same swizzled byte layout as load_tile gives).
template <int D>
struct OutCfg {
  static constexpr int TILE = BLK * D * 2;
  static constexpr int PT = BLK * BLK * 2;  // fp16 probabilities of one block
  static constexpr size_t k = TILE;                              // 2 key stages
  static constexpr size_t v = 3 * static_cast<size_t>(TILE);     // 2 value stages
  static constexpr size_t p = 5 * static_cast<size_t>(TILE);     // 2 probability tiles
  static constexpr size_t bars = p + 2 * static_cast<size_t>(PT);  // S[2], O, drain
  static constexpr size_t tslot = bars + 32;
  static constexpr size_t bytes = tslot + 16 + 1024;
};
constexpr uint32_t kOutTmemCols = 512;  // two 128-column logit blocks + O (D <= 128 columns)

// D[tmem] (+)= P[128 x 128 keys] * V[128 keys x D].
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, const unsigned char* p, const unsigned char* v, bool acc) {
  constexpr uint32_t idesc = tc::idesc_f16_f32_bmn(BLK, D);
  const uint32_t sp = smem_u32(p), sv = smem_u32(v);
#pragma unroll
  for (int ks = 0; ks < BLK / 16; ++ks) {
    const uint32_t aoff = static_cast<uint32_t>((ks >> 2) * (BLK * 128) + (ks & 3) * 32);
    tc::mma_f16(d_tmem, tc::desc_k_sw128(sp + aoff), tc::desc_mn_sw128(sv + ks * 2048u, BLK * 128), idesc,
                acc || ks > 0);
  }
}

__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity, int lane, int* err) {
  const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, kWaitLimit));
  if (!ok && lane == 0 && err) atomicOr(err, ERR_MMA_TIMEOUT);
  return ok;
}

template <int D>
__global__ void __launch_bounds__(NT, 1) out_tc(const PrefillParams prm) {
  using Cfg = OutCfg<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  unsigned char* sQ = smem;
  unsigned char* sK = smem + Cfg::k;
  unsigned char* sV = smem + Cfg::v;
  unsigned char* sP = smem + Cfg::p;
  uint64_t* mbS = reinterpret_cast<uint64_t*>(smem + Cfg::bars);
  uint64_t* mbO = mbS + 2;
  uint64_t* mbD = mbS + 3;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + Cfg::tslot);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = prm.L, pair = blockIdx.y;
  const int qb = gridDim.x - 1 - blockIdx.x;  // longest rows first
  const size_t base = static_cast<size_t>(pair) * L * D;
  const __half* Q = static_cast<const __half*>(prm.q) + base;
  const __half* K = static_cast<const __half*>(prm.k) + base;
  const __half* V = static_cast<const __half*>(prm.v) + base;
  const int n = qb + 1;
  const int quarter = warp & 3, half = warp >> 2;
  const int rl = quarter * 32 + lane, row = qb * BLK + rl;  // this thread's TMEM lane / query row

  griddep_wait();
  if (warp == 0) tc::tmem_alloc(tslot, kOutTmemCols);
  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(&mbS[i], 1);
    fence_mbar_init();
  }
  const float lse = lse_at(prm.lse2 + static_cast<size_t>(pair) * L, qb * BLK, rl, L);
  load_tile<D>(sQ, Q, qb * BLK, L, tid);
  load_tile<D>(sK, K, 0, L, tid);
  if (n > 1) load_tile<D>(sK + Cfg::TILE, K, BLK, L, tid);
  load_tile<D>(sV, V, 0, L, tid);
  cp_async_commit();
  cp_async_wait<0>();
  fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tslot;
  const uint32_t o_tmem = tbase + 2 * BLK;
  if (tid == 0) {
    issue_block<D>(tbase, sQ, sK);
    tc::mma_commit(&mbS[0]);
    if (n > 1) {
      issue_block<D>(tbase + BLK, sQ, sK + Cfg::TILE);
      tc::mma_commit(&mbS[1]);
    }
  }
  const uint32_t lane_addr = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
  bool ok = true;
  for (int j = 0; j < n; ++j) {
    const int b = j & 1;
    if (ok) ok = wait_all(&mbS[b], static_cast<uint32_t>((j >> 1) & 1), lane, prm.err);
    tc::fence_after_sync();
    if (j + 2 < n) load_tile<D>(sK + b * Cfg::TILE, K, (j + 2) * BLK, L, tid);  // S(j) has read stage b
    cp_async_commit();
    uint32_t ph[32];  // this thread's 64 probabilities as fp16 pairs
    if (ok) {
      float v[64];
      tc::tmem_ld32(lane_addr + static_cast<uint32_t>(b * BLK + half * 64), *reinterpret_cast<float(*)[32]>(v));
      tc::tmem_ld32(lane_addr + static_cast<uint32_t>(b * BLK + half * 64 + 32),
                    *reinterpret_cast<float(*)[32]>(v + 32));
      if (j == qb) {  // diagonal block: key half * 64 + e is visible to row rl if it is <= rl
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float p0 = half * 64 + 2 * e <= rl ? ex2(fmaf(v[2 * e], prm.qscale, -lse)) : 0.f;
          const float p1 = half * 64 + 2 * e + 1 <= rl ? ex2(fmaf(v[2 * e + 1], prm.qscale, -lse)) : 0.f;
          ph[e] = tc::cvt_half2(p0, p1);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          ph[e] = tc::cvt_half2(ex2(fmaf(v[2 * e], prm.qscale, -lse)), ex2(fmaf(v[2 * e + 1], prm.qscale, -lse)));
      }
    }
    // O(j-1) complete: probability tile b (last read by O(j-2)) and value
    // stage (j+1)%2 (read by O(j-1)) are free
    if (ok && j >= 1) ok = wait_all(mbO, static_cast<uint32_t>((j - 1) & 1), lane, prm.err);
    tc::fence_after_sync();
    if (j + 1 < n) load_tile<D>(sV + ((j + 1) & 1) * Cfg::TILE, V, (j + 1) * BLK, L, tid);
    cp_async_commit();
    if (ok) {
      unsigned char* prow = sP + b * Cfg::PT + half * (BLK * 128) + rl * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(prow + ((c ^ (rl & 7)) << 4)) = make_uint4(ph[4 * c], ph[4 * c + 1], ph[4 * c + 2],
                                                                            ph[4 * c + 3]);
    }
    cp_async_wait<1>();  // all but the value block j + 1 just requested
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();  // P(j) written, V(j) and K(j + 2) landed, S(j) read
    tc::fence_after_sync();
    if (tid == 0 && ok) {
      issue_pv<D>(o_tmem, sP + b * Cfg::PT, sV + b * Cfg::TILE, j > 0);
      tc::mma_commit(mbO);
      if (j + 2 < n) {
        issue_block<D>(tbase + b * BLK, sQ, sK + b * Cfg::TILE);
        tc::mma_commit(&mbS[b]);
      }
    }
  }
  if (ok) ok = wait_all(mbO, static_cast<uint32_t>((n - 1) & 1), lane, prm.err);
  tc::fence_after_sync();
  griddep_launch();
  if (ok) {
    float* dst = prm.out + (static_cast<size_t>(pair) * L + row) * D + half * (D / 2);
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      float o[32];
      tc::tmem_ld32(lane_addr + 2 * BLK + static_cast<uint32_t>(half * (D / 2) + c * 32), o);
      if (row < L) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
          reinterpret_cast<float4*>(dst + c * 32)[e] = make_float4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
      }
    }
  }
  // every MMA this CTA issued has completed before its TMEM is freed
  if (tid == 0) {
    tc::mma_commit(mbD);
    if (!mbar_wait_bounded(mbD, 0, kWaitLimit) && prm.err) atomicOr(prm.err, ERR_MMA_TIMEOUT);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_free(tbase, kOutTmemCols);
}

template <typename Kern>
cudaError_t launch_tc(Kern kern, dim3 grid, size_t smem, cudaStream_t s, const PrefillParams& prm) {
  cudaError_t e = kernel_attrs(reinterpret_cast<const void*>(kern), smem, false);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(NT);
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

cudaError_t launch_prefill_colsum_tc(const PrefillParams& prm, int D, int pairs, cudaStream_t s) {
  if (prm.L <= 0) return cudaSuccess;
  const dim3 grid((prm.L + BLK - 1) / BLK, pairs);
  if (D == 128) return launch_tc(colsum_tc<128>, grid, TcCfg<128>::bytes, s, prm);
  if (D == 64) return launch_tc(colsum_tc<64>, grid, TcCfg<64>::bytes, s, prm);
  return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_stats_tc(const PrefillParams& prm, int D, int pairs, cudaStream_t s) {
  if (prm.L <= 0) return cudaSuccess;
  if (D != 64 && D != 128) return cudaErrorInvalidValue;
  const dim3 grid((prm.L + BLK - 1) / BLK, pairs);
  cudaError_t e = D == 128 ? launch_tc(stats_tc<128>, grid, TcCfg<128>::bytes, s, prm)
                           : launch_tc(stats_tc<64>, grid, TcCfg<64>::bytes, s, prm);
  if (e != cudaSuccess || prm.out == nullptr) return e;
  return D == 128 ? launch_tc(out_tc<128>, grid, OutCfg<128>::bytes, s, prm)
                  : launch_tc(out_tc<64>, grid, OutCfg<64>::bytes, s, prm);
}

}  // namespace h2o
