// H2O prefill on the 5th-generation tensor cores (tcgen05, accumulators in
// tensor memory) for fp16 K/V: the row log-sum-exp pass, the attention
// output pass and the column-sum pass.
//
// Method: "H2O: Heavy-Hitter Oracle ... 深度解读报告", section 3.4 (prefill
// keep rule) with the score of section 3.3 / 2.3: every prompt token's score
// is the attention mass it receives, colsum_j = sum_{i>=j} exp(s_ij - lse_i),
// s_ij = scale * q_i . k_j; the output is ordinary causal attention,
// O_i = sum_j exp(s_ij - lse_i) v_j.
//
// All three passes work on 128 x 128 blocks of logits and are warp
// specialised.  Warp 0 streams operand tiles with TMA (3-D tensor maps over
// [P, L, D], 64-element boxes in the 128-byte swizzle that the MMAs read;
// rows past the prompt arrive as zeros) through rings of shared-memory
// stages; one lane of warp 1 issues tcgen05.mma (M = N = 128, K = 16, fp32
// accumulators in TMEM, two logit accumulators so the tensor core works on
// block i+1 while block i is exponentiated); eight compute warps read the
// accumulators with tcgen05.ld and do the exponentials.  Every hand-over is
// an mbarrier (TMA bytes, tcgen05.commit, or one arrive per compute warp), so
// no block-wide barrier sits in the streaming loops.
//  - rows (stats_tc): A = 128 query rows, B = key blocks 0..diagonal; TMEM
//    lane = query row; each compute thread keeps an online max / sum over
//    half of its row's columns.
//  - output (out_tc): with lse known, P = exp2(s - lse) needs no rescaling;
//    the compute warps store P as fp16 into TMEM (tcgen05.st) and the tensor
//    core accumulates O += P V in TMEM with A = P taken from TMEM and V as
//    stored ([key][d]) the MN-major B operand in shared memory.
//  - columns (colsum_tc): A = 128 keys, B = query blocks from the diagonal
//    down, i.e. the transposed logits; TMEM lane = key, so each thread sums
//    the probabilities its key receives with no cross-thread reduction
//    (float32 within a block, float64 across blocks: fixed order).
// Every wait is bounded; on a timeout the role stops, sets a device error
// bit, and the CTA still drains its copies and MMAs and frees its TMEM.
#include <cuda.h>  // CUtensorMap and the encoder's argument types (the encoder is looked up at run time)
#include <cuda_fp16.h>

#include <mutex>

#include "h2o_internal.cuh"
#include "ptx.cuh"

namespace h2o {
namespace {

constexpr float kNeg = -3.0e38f;
constexpr uint32_t kWaitLimit = 200000u;  // polls of <= 1 us: waits on this CTA's own copies and MMAs
constexpr int BLK = 128;                   // rows / columns of a logits block
constexpr int NCOMP = 8;                   // compute warps: 4 TMEM lane quarters x 2 column halves
constexpr int NT = (2 + NCOMP) * 32;       // + the TMA warp and the MMA warp
constexpr int kCompBar = 1;                // named barrier of the compute warps
// The output pass gives each compute warp a quarter of a block's columns (16
// warps: four per TMEM lane quarter), so that more warps hide the latency
// of its per-block chain (TMEM load, exponentials, reductions, TMEM store).
constexpr int NCOMP_O = 16;
constexpr int NT_O = (2 + NCOMP_O) * 32;

// Log2-domain lse of query row row0 + t; rows past the prompt get a huge
// value so that their probabilities exp2(s - lse) vanish without a mask.  A
// plain load: the rows of the vector need not be 16-byte aligned.
constexpr float kHugeLse = 3.0e38f;
__device__ __forceinline__ float lse_at(const float* src, int row0, int t, int L) {
  return row0 + t < L ? src[row0 + t] : kHugeLse;
}

// Kernel arguments: the pointers and sizes plus a tensor map per input.
struct TcArgs {
  CUtensorMap q, k, v;  // [P, L, D] fp16, box 64 x 128 x 1, 128-byte swizzle
  CUtensorMap o;        // [P, L, D] fp32 output, box 32 x 128 x 1, 128-byte swizzle
  PrefillParams prm;
};

template <int D>
struct Tile {
  static constexpr int BYTES = BLK * D * 2;  // a 128-row operand tile
  static constexpr int KB = BLK * 128;       // bytes of one 64-element K block of it
};

// 128 rows (row0..) of one pair's [L, D] matrix into a K-major tile: K block
// kb (64 elements) at tile + kb * 16 KB, row r at + r * 128 B, 16-byte chunk
// c at chunk c ^ (r % 8) (the TMA 128-byte swizzle; the tile is 1024-byte
// aligned).  Issued by one thread; completes Tile<D>::BYTES on `bar`.
template <int D>
__device__ __forceinline__ void tma_tile(unsigned char* tile, const CUtensorMap* map, int row0, int pair,
                                         uint64_t* bar) {
#pragma unroll
  for (int kb = 0; kb < D / 64; ++kb) tc::tma_load_3d(tile + kb * Tile<D>::KB, map, kb * 64, row0, pair, bar);
}

// D[tmem] = A[128 x D] * B[128 x D]^T over the head dimension (both K-major).
template <int D>
__device__ __forceinline__ void issue_block(uint32_t d_tmem, const unsigned char* a, const unsigned char* b) {
  constexpr uint32_t idesc = tc::idesc_f16_f32(BLK, BLK);
  const uint32_t sa = smem_u32(a), sb = smem_u32(b);
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const uint32_t off = static_cast<uint32_t>((ks >> 2) * Tile<D>::KB + (ks & 3) * 32);
    tc::mma_f16(d_tmem, tc::desc_k_sw128(sa + off), tc::desc_k_sw128(sb + off), idesc, ks > 0);
  }
}

// The swizzle is a function of address bits 4..9, so operand tiles start on
// a 1024-byte boundary of the shared window.
__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
  return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
}

// Bounded wait by one thread; a timeout latches the error bit.
__device__ __forceinline__ bool wait1(uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_wait_bounded(bar, parity, kWaitLimit)) return true;
  if (err) atomicOr(err, ERR_MMA_TIMEOUT);
  return false;
}
// Bounded wait by a whole warp; the result is warp-uniform, so the
// .sync.aligned TMEM loads that follow never diverge.
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, int lane, int* err) {
  const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, kWaitLimit));
  if (!ok && lane == 0 && err) atomicOr(err, ERR_MMA_TIMEOUT);
  return ok;
}

// A ring of N operand stages fed by TMA: use number u goes to stage u % N.
template <int N>
struct Ring {
  uint64_t* full;   // [N] producer -> consumer (TMA bytes)
  uint64_t* empty;  // [N] consumer -> producer
  // producer: wait until stage u % N is free again (its previous use released)
  __device__ bool acquire(int u, int* err) const {
    return u < N || wait1(&empty[u % N], static_cast<uint32_t>((u / N - 1) & 1), err);
  }
  __device__ uint64_t* full_of(int u) const { return &full[u % N]; }
  __device__ static uint32_t parity(int u) { return static_cast<uint32_t>((u / N) & 1); }
  // producer, at exit: every issued copy has landed (uses 0..issued-1)
  __device__ void drain(int issued, int* err) const {
    for (int u = issued - N > 0 ? issued - N : 0; u < issued; ++u) wait1(&full[u % N], parity(u), err);
  }
};

// Teardown: the MMA lane waits for all its MMAs, every thread meets, and
// warp 1 (which allocated them) frees the TMEM columns.
__device__ __forceinline__ void tmem_teardown(int warp, int lane, uint64_t* drain, uint32_t tbase, uint32_t cols,
                                              int* err) {
  if (warp == 1 && lane == 0) {
    tc::mma_commit(drain);
    wait1(drain, 0, err);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_free(tbase, cols);
}

// Set-up shared by the kernels: barrier init by one thread, TMEM allocation
// by warp 1, and the allocation's address published to every thread.
__device__ __forceinline__ uint32_t setup(int warp, uint64_t* bars, const uint32_t* counts, int nbars,
                                          uint32_t* tslot, uint32_t cols) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < nbars; ++i) mbar_init(&bars[i], counts[i]);
    fence_mbar_init();
  }
  if (warp == 1) tc::tmem_alloc(tslot, cols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  return *tslot;
}

// ------------------------------------------------------- row log-sum-exp
template <int D>
struct StatsCfg {
  static constexpr int NS = 2;  // key stages
  static constexpr size_t q = 0, k = Tile<D>::BYTES;
  static constexpr size_t bars = k + NS * static_cast<size_t>(Tile<D>::BYTES);
  static constexpr int NB = 10;  // qfull, kfull[2], kempty[2], sfull[2], sempty[2], drain
  static constexpr size_t tslot = bars + 8 * NB;
  static constexpr size_t red = (tslot + 16 + 15) / 16 * 16;  // [128] (m, l) of the upper column half
  static constexpr size_t bytes = red + BLK * 8 + 1024;       // + alignment slack
};

template <int D>
__global__ void __launch_bounds__(NT, 2) stats_tc(const __grid_constant__ TcArgs a) {
  using Cfg = StatsCfg<D>;
  constexpr int NS = Cfg::NS, TB = Tile<D>::BYTES;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  unsigned char* sQ = smem + Cfg::q;
  unsigned char* sK = smem + Cfg::k;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::bars);
  uint64_t* qfull = bars;
  const Ring<NS> kr{bars + 1, bars + 3};
  uint64_t* sfull = bars + 5;
  uint64_t* sempty = bars + 7;
  uint64_t* drain = bars + 9;
  float2* red = reinterpret_cast<float2*>(smem + Cfg::red);
  const PrefillParams& prm = a.prm;
  int* err = prm.err;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = prm.L, pair = blockIdx.y;
  const int qb = gridDim.x - 1 - blockIdx.x;  // longest rows first
  const int n = qb + 1;                      // key blocks 0..qb (causal)
  const uint32_t counts[Cfg::NB] = {1, 1, 1, 1, 1, 1, 1, NCOMP, NCOMP, 1};

  if (threadIdx.x == 0) {
    tc::prefetch_tensormap(&a.q);
    tc::prefetch_tensormap(&a.k);
  }
  griddep_wait();
  const int Lp = pair_len(prm.lens, prm.heads, L, pair);  // this pair's prompt length (L: row stride)
  if (qb * BLK >= Lp) return;                              // no rows of this pair here
  const uint32_t tbase = setup(warp, bars, counts, Cfg::NB, reinterpret_cast<uint32_t*>(smem + Cfg::tslot), 256);
  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      mbar_arrive_expect_tx(qfull, TB);
      tma_tile<D>(sQ, &a.q, qb * BLK, pair, qfull);
      int u = 0;
      for (; u < n && kr.acquire(u, err); ++u) {
        mbar_arrive_expect_tx(kr.full_of(u), TB);
        tma_tile<D>(sK + (u % NS) * TB, &a.k, u * BLK, pair, kr.full_of(u));
      }
      kr.drain(u, err);
      wait1(qfull, 0, err);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      bool ok = wait1(qfull, 0, err);
      for (int j = 0; ok && j < n; ++j) {
        const int b = j & 1;
        ok = wait1(kr.full_of(j), kr.parity(j), err) &&
             (j < 2 || wait1(&sempty[b], static_cast<uint32_t>(((j - 2) >> 1) & 1), err));
        if (!ok) break;
        tc::fence_after_sync();
        issue_block<D>(tbase + b * BLK, sQ, sK + (j % NS) * TB);
        tc::mma_commit(&sfull[b]);
        tc::mma_commit(&kr.empty[j % NS]);
      }
    }
    __syncwarp();
  } else {  // compute warps
    const int quarter = warp & 3, half = (warp - 2) >> 2;
    const int rl = quarter * 32 + lane, row = qb * BLK + rl;  // TMEM lane = query row
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    float m = kNeg, l = 0.f;
    for (int j = 0; j < n; ++j) {
      const int b = j & 1;
      if (!wait_warp(&sfull[b], static_cast<uint32_t>((j >> 1) & 1), lane, err)) break;
      tc::fence_after_sync();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int col0 = half * 64 + c * 32;
        float v[32];
        tc::tmem_ld32(lane_addr + static_cast<uint32_t>(b * BLK + col0), v);
        if (c == 1) {  // both loads of block j are done: accumulator b may take S(j+2)
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive_plain(&sempty[b]);
        }
        if (j == qb) {  // diagonal block: key col0 + e is visible to row rl if it is <= rl
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = col0 + e <= rl ? v[e] : -INFINITY;
        }
        // the max of the raw logits (scale > 0 commutes with max), two
        // chains of three-input maxima
        float c0 = max3(v[0], v[1], v[2]), c1 = v[3];
#pragma unroll
        for (int e = 4; e < 32; e += 4) {
          c0 = max3(c0, v[e], v[e + 1]);
          c1 = max3(c1, v[e + 2], v[e + 3]);
        }
        const float mn = fmaxf(m, fmaxf(c0, c1) * prm.qscale);
        // exp2(v * qscale - mn) summed, two columns per f32x2 FMA / add
        const uint64_t qs2 = f2_pack(prm.qscale, prm.qscale), nm2 = f2_pack(-mn, -mn);
        uint64_t s0 = 0, s1 = 0;  // packed (0.f, 0.f)
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          float x0, x1, x2, x3;
          f2_unpack(f2_fma(f2_pack(v[e], v[e + 1]), qs2, nm2), x0, x1);
          f2_unpack(f2_fma(f2_pack(v[e + 2], v[e + 3]), qs2, nm2), x2, x3);
          s0 = f2_add(s0, f2_pack(ex2(x0), ex2(x1)));
          s1 = f2_add(s1, f2_pack(ex2(x2), ex2(x3)));
        }
        float a0, a1, a2, a3;
        f2_unpack(s0, a0, a1);
        f2_unpack(s1, a2, a3);
        l = l * ex2(m - mn) + ((a0 + a1) + (a2 + a3));
        m = mn;
      }
    }
    // merge the two column halves of each row
    if (half == 1) red[rl] = make_float2(m, l);
    tc::named_sync(kCompBar, NCOMP * 32);
    if (half == 0 && row < Lp) {
      const float2 o = red[rl];
      const float M = fmaxf(m, o.x);
      prm.lse2[static_cast<size_t>(pair) * L + row] = M + log2f(l * ex2(m - M) + o.y * ex2(o.x - M));
    }
    griddep_launch();
  }
  tmem_teardown(warp, lane, drain, tbase, 256, err);
}

// ------------------------------------------------------- attention output
template <int D>
struct OutCfg {
  static constexpr int NK = 3, NV = 3;  // key / value stages
  static constexpr size_t q = 0, k = Tile<D>::BYTES;
  static constexpr size_t v = k + NK * static_cast<size_t>(Tile<D>::BYTES);
  static constexpr size_t bars = v + NV * static_cast<size_t>(Tile<D>::BYTES);
  // qfull, kfull[3], kempty[3], vfull[3], vempty[3], sfull[2], pfull[2], pempty[2], ofull, drain,
  // sempty[2]
  static constexpr int NB = 23;
  static constexpr size_t tslot = bars + 8 * NB;
  static constexpr size_t bytes = tslot + 16 + 1024;
};
// TMEM columns: two 128-column logit blocks, O (D <= 128 columns), and two
// 64-column fp16 probability blocks (P(j) is the A operand of O += P V)
constexpr uint32_t kOutTmemCols = 512;
constexpr uint32_t kOcol = 2 * BLK, kPcol = 3 * BLK;

// D[tmem] (+)= P[128 x 128 keys, in TMEM] * V[128 keys x D, MN-major in smem].
template <int D>
__device__ __forceinline__ void issue_pv_t(uint32_t d_tmem, uint32_t p_tmem, const unsigned char* v, bool acc) {
  constexpr uint32_t idesc = tc::idesc_f16_f32_bmn(BLK, D);
  const uint32_t sv = smem_u32(v);
#pragma unroll
  for (int ks = 0; ks < BLK / 16; ++ks)  // 16 keys = 8 packed columns per step
    tc::mma_f16_ta(d_tmem, p_tmem + ks * 8, tc::desc_mn_sw128(sv + ks * 2048u, BLK * 128), idesc, acc || ks > 0);
}

template <int D>
__global__ void __launch_bounds__(NT_O, 1) out_tc(const __grid_constant__ TcArgs a) {
  using Cfg = OutCfg<D>;
  constexpr int NK = Cfg::NK, NV = Cfg::NV, TB = Tile<D>::BYTES;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  unsigned char* sQ = smem + Cfg::q;
  unsigned char* sK = smem + Cfg::k;
  unsigned char* sV = smem + Cfg::v;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::bars);
  uint64_t* qfull = bars;
  const Ring<NK> kr{bars + 1, bars + 1 + NK};
  const Ring<NV> vr{bars + 1 + 2 * NK, bars + 1 + 2 * NK + NV};
  uint64_t* sfull = bars + 1 + 2 * NK + 2 * NV;
  uint64_t* pfull = sfull + 2;
  uint64_t* pempty = sfull + 4;
  uint64_t* ofull = sfull + 6;
  uint64_t* drain = sfull + 7;
  uint64_t* sempty = sfull + 8;
  static_assert(1 + 2 * NK + 2 * NV + 10 == Cfg::NB, "barrier count");
  const PrefillParams& prm = a.prm;
  int* err = prm.err;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = prm.L, pair = blockIdx.y;
  const int qb = gridDim.x - 1 - blockIdx.x;  // longest rows first
  const int n = qb + 1;
  // qfull, K full/empty, V full/empty, sfull[2]: one arrival (TMA or commit);
  // pfull[2], sempty[2]: one per compute warp; pempty[2], ofull, drain: a commit
  uint32_t counts[Cfg::NB];
#pragma unroll
  for (int i = 0; i < Cfg::NB; ++i) {
    const int r = i - (1 + 2 * NK + 2 * NV);  // index from sfull[0]
    counts[i] = (r == 2 || r == 3 || r == 8 || r == 9) ? NCOMP_O : 1;
  }

  if (threadIdx.x == 0) {
    tc::prefetch_tensormap(&a.q);
    tc::prefetch_tensormap(&a.k);
    tc::prefetch_tensormap(&a.v);
    tc::prefetch_tensormap(&a.o);
  }
  griddep_wait();
  const int Lp = pair_len(prm.lens, prm.heads, L, pair);  // this pair's prompt length (L: row stride)
  if (qb * BLK >= Lp) return;
  const uint32_t tbase =
      setup(warp, bars, counts, Cfg::NB, reinterpret_cast<uint32_t*>(smem + Cfg::tslot), kOutTmemCols);
  const uint32_t o_tmem = tbase + kOcol;
  if (warp == 0) {
    if (lane == 0) {  // TMA producer, in the order the MMAs consume: K0 K1 K2 V0 K3 V1 ...
      mbar_arrive_expect_tx(qfull, TB);
      tma_tile<D>(sQ, &a.q, qb * BLK, pair, qfull);
      int uk = 0, uv = 0;
      auto issue_k = [&](int j) {
        if (!kr.acquire(j, err)) return false;
        mbar_arrive_expect_tx(kr.full_of(j), TB);
        tma_tile<D>(sK + (j % NK) * TB, &a.k, j * BLK, pair, kr.full_of(j));
        uk = j + 1;
        return true;
      };
      auto issue_v = [&](int j) {
        if (!vr.acquire(j, err)) return false;
        mbar_arrive_expect_tx(vr.full_of(j), TB);
        tma_tile<D>(sV + (j % NV) * TB, &a.v, j * BLK, pair, vr.full_of(j));
        uv = j + 1;
        return true;
      };
      bool ok = issue_k(0) && (n < 2 || issue_k(1));
      for (int j = 0; ok && j < n; ++j) ok = (j + 2 >= n || issue_k(j + 2)) && issue_v(j);
      kr.drain(uk, err);
      vr.drain(uv, err);
      wait1(qfull, 0, err);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer: S0 S1, then per block j: S(j+2) once S(j) is read, O(j) once P(j) is in
      bool ok = wait1(qfull, 0, err);
      for (int j = 0; ok && j < 2 && j < n; ++j) {
        ok = wait1(kr.full_of(j), kr.parity(j), err);
        if (!ok) break;
        tc::fence_after_sync();
        issue_block<D>(tbase + j * BLK, sQ, sK + (j % NK) * TB);
        tc::mma_commit(&sfull[j]);
        tc::mma_commit(&kr.empty[j % NK]);
      }
      for (int j = 0; ok && j < n; ++j) {
        const int b = j & 1;
        const uint32_t ph = static_cast<uint32_t>((j >> 1) & 1);
        if (j + 2 < n) {  // every compute warp has loaded S(j): accumulator b takes S(j+2)
          ok = wait1(&sempty[b], ph, err) && wait1(kr.full_of(j + 2), kr.parity(j + 2), err);
          if (!ok) break;
          tc::fence_after_sync();
          issue_block<D>(tbase + b * BLK, sQ, sK + ((j + 2) % NK) * TB);
          tc::mma_commit(&sfull[b]);
          tc::mma_commit(&kr.empty[(j + 2) % NK]);
        }
        ok = wait1(&pfull[b], ph, err) && wait1(vr.full_of(j), vr.parity(j), err);
        if (!ok) break;
        tc::fence_after_sync();
        issue_pv_t<D>(o_tmem, tbase + kPcol + b * 64, sV + (j % NV) * TB, j > 0);
        tc::mma_commit(&pempty[b]);
        tc::mma_commit(&vr.empty[j % NV]);
      }
      if (ok) tc::mma_commit(ofull);
    }
    __syncwarp();
  } else {  // compute warps: lane quarter (warp % 4) x column part (32 of the 128)
    const int quarter = warp & 3, part = (warp - 2) >> 2;
    const int rl = quarter * 32 + lane;  // O readout: TMEM lane = query row qb * BLK + rl
    const int col0 = part * 32;          // this warp's keys in a block / its O columns
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    // Logits are read in the 16x256b shape, two loads per block (lane halves
    // h = 0, 1 of the quarter): element e of repetition k of half h holds
    // row r4 + 16h + 8(e >> 1) and key k4 + 8k + (e & 1).  Each thread thus
    // holds 4 rows x 8 keys, and a key's 32 rows of the quarter sit in the 8
    // lanes that share lane % 4.
    const int r4 = quarter * 32 + (lane >> 2);
    const int k4 = col0 + 2 * (lane & 3);
    float nlse[4];  // -lse of row r4 + 8i, i = 2h + (e >> 1)
#pragma unroll
    for (int i = 0; i < 4; ++i) nlse[i] = -lse_at(prm.lse2 + static_cast<size_t>(pair) * L, qb * BLK, r4 + 8 * i, Lp);
    // this pair's column-sum partials: one 4 x 128-float row per (query block, key block <= it)
    float* cs_part = prm.cs_part ? prm.cs_part + static_cast<size_t>(pair) * colsum_partial_floats(L, 1) : nullptr;
    const uint64_t qs2 = f2_pack(prm.qscale, prm.qscale);
    const uint32_t half_hi = 16u << 16;  // TMEM lane offset of the upper half
    bool ok = true;
    for (int j = 0; ok && j < n; ++j) {
      const int b = j & 1;
      ok = wait_warp(&sfull[b], static_cast<uint32_t>((j >> 1) & 1), lane, err);
      if (!ok) break;
      tc::fence_after_sync();
      uint32_t raw[2][16];
      const uint32_t sa = lane_addr + static_cast<uint32_t>(b * BLK + col0);
      tc::tmem_ld_16x256b_x4_pair(sa, sa + half_hi, raw[0], raw[1]);
      // accumulator b may take the next logit block as soon as every compute
      // warp has its slice in registers
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_plain(&sempty[b]);
      float v[2][16];  // probabilities, same element order as raw
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            const int i = 2 * h + g, e = 4 * k + 2 * g;
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(raw[h][e]), __uint_as_float(raw[h][e + 1])), qs2,
                             f2_pack(nlse[i], nlse[i])),
                      x0, x1);
            v[h][e] = ex2(x0);
            v[h][e + 1] = ex2(x1);
          }
      if (j == qb) {  // diagonal block: key k is visible to row r if k <= r
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (k4 + 8 * k + (e & 1) > r4 + 16 * h + 8 * (e >> 1)) v[h][4 * k + e] = 0.f;
      }
      // probability block b (TMEM) was last read by O(j-2).  Keys k4 + 8k and
      // k4 + 8k + 1 of a row are one fp16 pair, packed column col0/2 + 4k +
      // lane % 4: the 16x128b store puts element g of repetition k there, in
      // row r4 + 16h + 8g.
      uint32_t ph[2][8];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int g = 0; g < 2; ++g) ph[h][2 * k + g] = tc::cvt_half2(v[h][4 * k + 2 * g], v[h][4 * k + 2 * g + 1]);
      if (j >= 2 && !(ok = wait_warp(&pempty[b], static_cast<uint32_t>(((j - 2) >> 1) & 1), lane, err))) break;
      const uint32_t pa = lane_addr + kPcol + static_cast<uint32_t>(b * 64 + col0 / 2);
      tc::tmem_st_16x128b_x4(pa, ph[0]);
      tc::tmem_st_16x128b_x4(pa + half_hi, ph[1]);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_plain(&pfull[b]);
      if (cs_part) {
        // while the tensor core works on P V: column sums over the quarter's
        // 32 rows.  Each thread adds its 4 rows of its 8 keys (c[2k + x] for
        // key k4 + 8k + x), then a reduce-scatter over the lanes sharing
        // lane % 4 leaves key index (lane >> 2) & 7 in each lane; one
        // 128-byte store per warp.
        float c[8];
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int x = 0; x < 2; ++x)
            c[2 * k + x] = (v[0][4 * k + x] + v[0][4 * k + 2 + x]) + (v[1][4 * k + x] + v[1][4 * k + 2 + x]);
#pragma unroll
        for (int off = 16, w = 4; off >= 4; off >>= 1, w >>= 1) {
          const bool hi = (lane & off) != 0;
#pragma unroll
          for (int i = 0; i < w; ++i) {
            const float keep = hi ? c[i + w] : c[i];
            const float send = hi ? c[i] : c[i + w];
            c[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
          }
        }
        const int c8 = (lane >> 2) & 7;
        cs_part[(static_cast<size_t>(qb) * (qb + 1) / 2 + j) * (4 * BLK) + quarter * BLK + k4 + 8 * (c8 >> 1) +
                (c8 & 1)] = c[0];
      }
    }
    ok = ok && wait_warp(ofull, 0, lane, err);
    tc::fence_after_sync();
    // O leaves through shared memory (the key ring is free once every MMA has
    // completed): boxes of 128 rows x 32 floats in the 128-byte swizzle (row
    // r's 16-byte chunk c at chunk c ^ (r % 8): conflict-free for a warp's 32
    // rows), written out by TMA stores clipped at the prompt's end.  Column
    // part p of O is box p.
    unsigned char* sO = sK;
    if (ok && col0 < D) {
      float o[32];
      tc::tmem_ld32(lane_addr + kOcol + static_cast<uint32_t>(col0), o);
      unsigned char* rowp = sO + part * (BLK * 128) + rl * 128;
#pragma unroll
      for (int e = 0; e < 8; ++e)
        *reinterpret_cast<float4*>(rowp + ((e ^ (rl & 7)) << 4)) =
            make_float4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
    }
    fence_proxy_async_smem();
    tc::named_sync(kCompBar, NCOMP_O * 32);
    if (warp == 2 && lane == 0) {
#pragma unroll
      for (int bx = 0; bx < D / 32; ++bx) tc::tma_store_3d(&a.o, sO + bx * (BLK * 128), bx * 32, qb * BLK, pair);
      tc::bulk_commit();
      tc::bulk_wait_read_all();  // shared memory stays valid until the stores have read it
    }
    griddep_launch();
  }
  tmem_teardown(warp, lane, drain, tbase, kOutTmemCols, err);
}

// ------------------------------------------------------------ column sums
template <int D>
struct ColCfg {
  static constexpr int NS = 2;  // query stages
  static constexpr size_t k = 0, q = Tile<D>::BYTES;
  static constexpr size_t lse = q + NS * static_cast<size_t>(Tile<D>::BYTES);  // [NCOMP][2][64] floats
  static constexpr size_t bars = lse + NCOMP * 2 * 64 * 4;
  static constexpr int NB = 10;  // kfull, qfull[2], qempty[2], sfull[2], sempty[2], drain
  static constexpr size_t tslot = bars + 8 * NB;
  static constexpr size_t red = (tslot + 16 + 15) / 16 * 16;  // [128] doubles of the upper column half
  static constexpr size_t bytes = red + BLK * 8 + 1024;
};

template <int D>
__global__ void __launch_bounds__(NT, 2) colsum_tc(const __grid_constant__ TcArgs a) {
  using Cfg = ColCfg<D>;
  constexpr int NS = Cfg::NS, TB = Tile<D>::BYTES;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  unsigned char* sK = smem + Cfg::k;
  unsigned char* sQ = smem + Cfg::q;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::bars);
  uint64_t* kfull = bars;
  const Ring<NS> qr{bars + 1, bars + 3};
  uint64_t* sfull = bars + 5;
  uint64_t* sempty = bars + 7;
  uint64_t* drain = bars + 9;
  double* red = reinterpret_cast<double*>(smem + Cfg::red);
  const PrefillParams& prm = a.prm;
  int* err = prm.err;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = prm.L, pair = blockIdx.y, kb = blockIdx.x;

  const uint32_t counts[Cfg::NB] = {1, 1, 1, 1, 1, 1, 1, NCOMP, NCOMP, 1};

  if (threadIdx.x == 0) {
    tc::prefetch_tensormap(&a.q);
    tc::prefetch_tensormap(&a.k);
  }
  griddep_wait();
  const int Lp = pair_len(prm.lens, prm.heads, L, pair);  // this pair's prompt length (L: row stride)
  const int n = (Lp + BLK - 1) / BLK - kb;                 // query blocks from the diagonal down
  if (n <= 0) return;
  const uint32_t tbase = setup(warp, bars, counts, Cfg::NB, reinterpret_cast<uint32_t*>(smem + Cfg::tslot), 256);
  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      mbar_arrive_expect_tx(kfull, TB);
      tma_tile<D>(sK, &a.k, kb * BLK, pair, kfull);
      int u = 0;
      for (; u < n && qr.acquire(u, err); ++u) {
        mbar_arrive_expect_tx(qr.full_of(u), TB);
        tma_tile<D>(sQ + (u % NS) * TB, &a.q, (kb + u) * BLK, pair, qr.full_of(u));
      }
      qr.drain(u, err);
      wait1(kfull, 0, err);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer: S^T(i) = K Q_i^T
      bool ok = wait1(kfull, 0, err);
      for (int i = 0; ok && i < n; ++i) {
        const int b = i & 1;
        ok = wait1(qr.full_of(i), qr.parity(i), err) &&
             (i < 2 || wait1(&sempty[b], static_cast<uint32_t>(((i - 2) >> 1) & 1), err));
        if (!ok) break;
        tc::fence_after_sync();
        issue_block<D>(tbase + b * BLK, sK, sQ + (i % NS) * TB);
        tc::mma_commit(&sfull[b]);
        tc::mma_commit(&qr.empty[i % NS]);
      }
    }
    __syncwarp();
  } else {  // compute warps
    const int cw = warp - 2, quarter = warp & 3, half = cw >> 2;
    const int kl = quarter * 32 + lane, key = kb * BLK + kl;  // TMEM lane = key
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    // this warp's 64 query columns' lse values, negated, one block ahead:
    // lane t fetches columns 2t, 2t + 1 of the next block while this one is
    // worked on
    const float* lse2 = prm.lse2 + static_cast<size_t>(pair) * L;
    float* wl = reinterpret_cast<float*>(smem + Cfg::lse) + cw * 128;  // [2][64]
    const int c0 = half * 64 + 2 * lane;
    wl[2 * lane] = -lse_at(lse2, kb * BLK, c0, Lp);
    wl[2 * lane + 1] = -lse_at(lse2, kb * BLK, c0 + 1, Lp);
    __syncwarp();
    double dacc = 0.0;
    for (int i = 0; i < n; ++i) {
      const int b = i & 1;
      float n0 = -kHugeLse, n1 = -kHugeLse;
      if (i + 1 < n) {
        n0 = -lse_at(lse2, (kb + i + 1) * BLK, c0, Lp);
        n1 = -lse_at(lse2, (kb + i + 1) * BLK, c0 + 1, Lp);
      }
      if (!wait_warp(&sfull[b], static_cast<uint32_t>((i >> 1) & 1), lane, err)) break;
      tc::fence_after_sync();
      const float* nlse = wl + b * 64;
      const uint64_t qs2 = f2_pack(prm.qscale, prm.qscale);
      float acc0 = 0.f, acc1 = 0.f;
      uint64_t acc2 = 0, acc3 = 0;  // packed (0.f, 0.f)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int col0 = half * 64 + c * 32;
        float v[32];
        tc::tmem_ld32(lane_addr + static_cast<uint32_t>(b * BLK + col0), v);
        const float4* l4 = reinterpret_cast<const float4*>(nlse + c * 32);
        if (i == 0) {  // diagonal block: query col0 + e sees key kl only if kl <= col0 + e
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 t = l4[j];
            const int e = 4 * j;
            acc0 += kl <= col0 + e ? ex2(fmaf(v[e], prm.qscale, t.x)) : 0.f;
            acc1 += kl <= col0 + e + 1 ? ex2(fmaf(v[e + 1], prm.qscale, t.y)) : 0.f;
            acc0 += kl <= col0 + e + 2 ? ex2(fmaf(v[e + 2], prm.qscale, t.z)) : 0.f;
            acc1 += kl <= col0 + e + 3 ? ex2(fmaf(v[e + 3], prm.qscale, t.w)) : 0.f;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 t = l4[j];
            const int e = 4 * j;
            // two columns per f32x2 FMA / add
            float x0, x1, x2, x3;
            f2_unpack(f2_fma(f2_pack(v[e], v[e + 1]), qs2, f2_pack(t.x, t.y)), x0, x1);
            f2_unpack(f2_fma(f2_pack(v[e + 2], v[e + 3]), qs2, f2_pack(t.z, t.w)), x2, x3);
            acc2 = f2_add(acc2, f2_pack(ex2(x0), ex2(x1)));
            acc3 = f2_add(acc3, f2_pack(ex2(x2), ex2(x3)));
          }
        }
      }
      float a0, a1, a2, a3;
      f2_unpack(acc2, a0, a1);
      f2_unpack(acc3, a2, a3);
      dacc += static_cast<double>((acc0 + acc1) + ((a0 + a1) + (a2 + a3)));
      tc::fence_before_sync();
      __syncwarp();  // also: every lane is done with lse slot b
      if (lane == 0) tc::mbar_arrive_plain(&sempty[b]);  // accumulator b may be overwritten
      wl[(b ^ 1) * 64 + 2 * lane] = n0;
      wl[(b ^ 1) * 64 + 2 * lane + 1] = n1;
      __syncwarp();
    }
    if (half == 1) red[kl] = dacc;
    tc::named_sync(kCompBar, NCOMP * 32);
    if (half == 0 && key < Lp) prm.colsum[static_cast<size_t>(pair) * L + key] = static_cast<float>(dacc + red[kl]);
    griddep_launch();
  }
  tmem_teardown(warp, lane, drain, tbase, 256, err);
}

// ------------------------------------------------- column sums from partials
// colsum_j = sum over query blocks qb >= j / 128 and the four TMEM lane
// quarters of the output pass's partial column sums (each a float32 sum over
// 32 rows), added in a fixed order (query blocks ascending, quarters 0..3)
// with Neumaier's compensated summation in float32 ("Rundungsfehleranalyse
// einiger Verfahren zur Summation endlicher Summen", 1974): the result is
// within about one float32 ulp of the exact sum of the partials.  GB300's
// float64 rate is a small fraction of its float32 rate, so plain float64
// accumulation made this kernel arithmetic-bound.  Four query blocks' loads
// are issued before they are added.
struct Neumaier {
  float s = 0.f, c = 0.f;  // running sum, accumulated rounding errors
  __device__ __forceinline__ void add(float x) {
    const float t = s + x;
    c += fabsf(s) >= fabsf(x) ? (s - t) + x : (x - t) + s;
    s = t;
  }
  __device__ __forceinline__ float value() const { return s + c; }
};

__global__ void __launch_bounds__(BLK) colsum_reduce_kernel(const PrefillParams prm) {
  griddep_wait();
  const int pair = blockIdx.y, kb = blockIdx.x, col = threadIdx.x;
  const int L = prm.L;
  const int Lp = pair_len(prm.lens, prm.heads, L, pair);
  const int nbp = (Lp + BLK - 1) / BLK;  // query blocks the output pass ran for this pair
  if (kb >= nbp) return;
  const float* part = prm.cs_part + static_cast<size_t>(pair) * colsum_partial_floats(L, 1) + col;
  auto row = [&](int qb) { return part + (static_cast<size_t>(qb) * (qb + 1) / 2 + kb) * (4 * BLK); };
  Neumaier acc;
  int qb = kb;
  for (; qb + 4 <= nbp; qb += 4) {
    float v[16];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float* r = row(qb + u);
#pragma unroll
      for (int h = 0; h < 4; ++h) v[4 * u + h] = __ldg(r + h * BLK);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) acc.add(v[i]);
  }
  for (; qb < nbp; ++qb) {
    const float* r = row(qb);
    float v[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) v[h] = __ldg(r + h * BLK);
#pragma unroll
    for (int h = 0; h < 4; ++h) acc.add(v[h]);
  }
  griddep_launch();
  const int key = kb * BLK + col;
  if (key < Lp) prm.colsum[static_cast<size_t>(pair) * L + key] = acc.value();
}

// ------------------------------------------------------------------ host
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime.
EncodeTiled encoder() {
  static const EncodeTiled fn = []() -> EncodeTiled {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return reinterpret_cast<EncodeTiled>(p);
  }();
  return fn;
}

// Tensor map of a [P, L, D] array (16-byte aligned) of fp16 (boxes 64 x 128
// x 1) or fp32 (boxes 32 x 128 x 1): 128-byte rows of a box, 128-byte
// swizzle, zeros past the ends on loads, clipping on stores.
bool encode_map(CUtensorMap* m, const void* base, int D, int L, int P, bool f32 = false) {
  const EncodeTiled enc = encoder();
  if (!enc || !base) return false;
  const cuuint64_t e = f32 ? 4 : 2;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(P)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * e, static_cast<cuuint64_t>(L) * D * e};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / e), BLK, 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base),
             dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename Kern>
cudaError_t launch_tc(Kern kern, dim3 grid, size_t smem, cudaStream_t s, const TcArgs& args, int threads = NT) {
  cudaError_t e = kernel_attrs(reinterpret_cast<const void*>(kern), smem, false);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args);
}

bool make_args(TcArgs& a, const PrefillParams& prm, int D, int pairs, bool with_v) {
  a = TcArgs{};
  a.prm = prm;
  return encode_map(&a.q, prm.q, D, prm.L, pairs) && encode_map(&a.k, prm.k, D, prm.L, pairs) &&
         (!with_v || (encode_map(&a.v, prm.v, D, prm.L, pairs) && encode_map(&a.o, prm.out, D, prm.L, pairs, true)));
}

}  // namespace

cudaError_t launch_prefill_stats_tc(const PrefillParams& prm, int D, int pairs, cudaStream_t s) {
  if (prm.L <= 0) return cudaSuccess;
  if (D != 64 && D != 128) return cudaErrorInvalidValue;
  TcArgs args;
  if (!make_args(args, prm, D, pairs, prm.out != nullptr)) return cudaErrorInvalidValue;
  const dim3 grid((prm.L + BLK - 1) / BLK, pairs);
  cudaError_t e = D == 128 ? launch_tc(stats_tc<128>, grid, StatsCfg<128>::bytes, s, args)
                           : launch_tc(stats_tc<64>, grid, StatsCfg<64>::bytes, s, args);
  if (e != cudaSuccess || prm.out == nullptr) return e;
  return D == 128 ? launch_tc(out_tc<128>, grid, OutCfg<128>::bytes, s, args, NT_O)
                  : launch_tc(out_tc<64>, grid, OutCfg<64>::bytes, s, args, NT_O);
}

cudaError_t launch_colsum_reduce(const PrefillParams& prm, int pairs, cudaStream_t s) {
  if (prm.L <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((prm.L + BLK - 1) / BLK, pairs);
  cfg.blockDim = dim3(BLK);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, colsum_reduce_kernel, prm);
}

cudaError_t launch_prefill_colsum_tc(const PrefillParams& prm, int D, int pairs, cudaStream_t s) {
  if (prm.L <= 0) return cudaSuccess;
  if (D != 64 && D != 128) return cudaErrorInvalidValue;
  TcArgs args;
  if (!make_args(args, prm, D, pairs, false)) return cudaErrorInvalidValue;
  const dim3 grid((prm.L + BLK - 1) / BLK, pairs);
  return D == 128 ? launch_tc(colsum_tc<128>, grid, ColCfg<128>::bytes, s, args)
                  : launch_tc(colsum_tc<64>, grid, ColCfg<64>::bytes, s, args);
}

}  // namespace h2o
