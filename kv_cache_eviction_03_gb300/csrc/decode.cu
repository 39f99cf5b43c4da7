// Fused H2O decode step: attention over the kept slots + the new token,
// accumulated-score update, eviction of the lowest (score, position) slot
// outside the recent window, in-place overwrite with the new K/V.
//
// Method: "H2O: Heavy-Hitter Oracle ... 深度解读报告", section 3.1 (softmax over
// kept entries only, one eviction per step), section 3.3 (Algorithm 1: the
// evicted entry minimises the accumulated attention score), section 3.4 (slot
// store preallocated and overwritten in place, recent region as a circular
// queue, one heavy hitter per head evicted per step).
//
// GB300 design.  Decode reads every kept K and V row once per step: about
// 1 FLOP per byte, so the kernel is bound by HBM bandwidth and uses no tensor
// cores.  One pair (batch row, head) is handled by a thread-block cluster of S
// CTAs; CTA r owns the contiguous slot range [r*chunk, (r+1)*chunk).  Each CTA
// streams its K and V rows through a ring of shared-memory stages filled by
// 1-D bulk async copies (cp.async.bulk, mbarrier completion) and keeps a
// base-2 online softmax (m, l, o) per row group.  The CTAs then exchange their
// partial (m, l, o) through distributed shared memory, so every CTA knows the
// pair's global max and normaliser without a second pass over K: each turns
// its own logits (kept in shared memory) into probabilities, adds them to its
// slots' scores, and proposes its lowest candidate key (score bits, position)
// packed in 64 bits (non-negative float bits order like the floats).  The
// cluster's minimum is the victim; the CTA that owns it writes the new row.
// Cluster barriers are hardware barriers of co-scheduled CTAs: no CTA spins
// on another.
#include <cooperative_groups.h>
#include <cuda_fp16.h>

#include "h2o_internal.cuh"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace h2o {
namespace {

constexpr float kNeg = -3.0e38f;  // finite "minus infinity" for running maxima
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr int kMaxChunk = 4096;

template <typename T, int D, int NT, int TILE, int NSTAGE>
struct DecodeCfg {
  static constexpr int E = sizeof(T);
  static constexpr int ROWB = D * E;    // bytes per K or V row
  static constexpr int EPV = 16 / E;    // elements per 16-byte vector
  static constexpr int LPR = ROWB / 16; // lanes per row
  static constexpr int RPI = 32 / LPR;  // rows per warp-wide load
  static constexpr int NW = NT / 32;
  static constexpr int RPW = TILE / NW; // rows per warp per tile
  static constexpr int IPW = RPW / RPI; // warp-wide loads per tile, per operand
  static constexpr int STAGE = 2 * TILE * ROWB;
  static_assert(LPR >= 1 && LPR <= 32, "row must be 16..512 bytes");
  static_assert(RPW % RPI == 0 && IPW >= 1, "tile must cover whole warp loads");
  static_assert(NT >= D, "one thread per output dimension in the merge");
};

struct __align__(16) Xch {
  float m, l, s_self, pad;
  unsigned long long key;
  int slot, pad2;
};

// Shared-memory layout; identical on host and device.
template <int D, int NW, int STAGE, int NSTAGE>
struct Layout {
  static constexpr size_t bars = 0;
  static constexpr size_t xch = 128;
  static constexpr size_t xo = xch + sizeof(Xch);  // cluster-visible partial o[D]
  static constexpr size_t red = (xo + D * 4 + 127) / 128 * 128;
  static constexpr size_t gm = red + NW * (D + 4) * 4;     // per-rank m / l / key / slot copies
  static constexpr size_t stages = (gm + 16 * 24 + 127) / 128 * 128;
  static constexpr size_t tail = stages + (size_t)NSTAGE * STAGE;  // then lg, sc, ps [chunk]
  static size_t bytes(int chunk) { return tail + (size_t)chunk * 12; }
};

template <typename T, int D, int NT, int TILE, int NSTAGE>
__global__ void __launch_bounds__(NT) decode_kernel(const DecodeParams prm) {
  using Cfg = DecodeCfg<T, D, NT, TILE, NSTAGE>;
  using Lay = Layout<D, Cfg::NW, Cfg::STAGE, NSTAGE>;
  constexpr int EPV = Cfg::EPV, LPR = Cfg::LPR, RPI = Cfg::RPI, IPW = Cfg::IPW, ROWB = Cfg::ROWB;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::bars);
  Xch* xch = reinterpret_cast<Xch*>(smem + Lay::xch);
  float* xo = reinterpret_cast<float*>(smem + Lay::xo);
  float* red = reinterpret_cast<float*>(smem + Lay::red);
  float* g_m = reinterpret_cast<float*>(smem + Lay::gm);
  float* g_l = g_m + 16;
  float* g_self = g_l + 16;  // [1] (padded to 16)
  unsigned long long* g_key = reinterpret_cast<unsigned long long*>(g_self + 16);
  int* g_slot = reinterpret_cast<int*>(g_key + 16);
  unsigned char* stage_base = smem + Lay::stages;
  float* lg = reinterpret_cast<float*>(smem + Lay::tail);
  float* sc = lg + prm.chunk;
  int* ps = reinterpret_cast<int*>(sc + prm.chunk);
  __shared__ unsigned long long blk_key[Cfg::NW];
  __shared__ int blk_slot;

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int S = static_cast<int>(cluster.num_blocks());
  const int pair = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = lane / LPR, lig = lane % LPR;

  griddep_wait();  // the previous step on this cache must be complete

  const PairCtr ctr = prm.ctr[pair];
  const int C = prm.C, R = prm.R;
  const int p = ctr.p, count = ctr.count, head = ctr.head;
  const bool full = count >= C;
  const int lo = rank * prm.chunk;
  const int hi = min(lo + prm.chunk, count);
  const int nrows = max(hi - lo, 0);
  const int ntiles = (nrows + TILE - 1) / TILE;
  const size_t slot0 = static_cast<size_t>(pair) * C + lo;
  const unsigned char* gK = static_cast<const unsigned char*>(prm.K) + slot0 * ROWB;
  const unsigned char* gV = static_cast<const unsigned char*>(prm.V) + slot0 * ROWB;

  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  uint64_t policy = 0;
  if (tid == 0) {
    policy = policy_evict_first();
    const int first = ntiles < NSTAGE ? ntiles : NSTAGE;
    for (int t = 0; t < first; ++t) {
      const int rows = min(TILE, nrows - t * TILE);
      const uint32_t bytes = static_cast<uint32_t>(rows * ROWB);
      unsigned char* st = stage_base + static_cast<size_t>(t) * Cfg::STAGE;
      mbar_arrive_expect_tx(&bars[t], 2 * bytes);
      bulk_g2s_stream(st, gK + static_cast<size_t>(t) * TILE * ROWB, bytes, &bars[t], policy);
      bulk_g2s_stream(st + TILE * ROWB, gV + static_cast<size_t>(t) * TILE * ROWB, bytes, &bars[t], policy);
    }
  }

  // q, pre-scaled so that exp2(logit) is the softmax numerator
  float qv[EPV];
  {
    const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(prm.q) +
                                                    static_cast<size_t>(pair) * ROWB + lig * 16);
    Vec16<T>::unpack(u, qv);
#pragma unroll
    for (int e = 0; e < EPV; ++e) qv[e] *= prm.qscale;
  }
  // scores and positions of this CTA's slots (needed after the softmax)
  for (int j = tid; j < nrows; j += NT) {
    sc[j] = prm.score[slot0 + j];
    ps[j] = prm.pos[slot0 + j];
  }

  float m = kNeg, l = 0.f, o[EPV];
#pragma unroll
  for (int e = 0; e < EPV; ++e) o[e] = 0.f;
  float s_self = 0.f;
  if (rank == 0 && warp == 0) {
    // the new token attends to itself: row group 0 of warp 0 starts from it
    float kf[EPV];
    const uint4 ku = *reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(prm.k_new) +
                                                     static_cast<size_t>(pair) * ROWB + lig * 16);
    Vec16<T>::unpack(ku, kf);
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < EPV; ++e) acc = fmaf(qv[e], kf[e], acc);
#pragma unroll
    for (int off = LPR / 2; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    s_self = acc;
    if (grp == 0) {
      const uint4 vu = *reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(prm.v_new) +
                                                       static_cast<size_t>(pair) * ROWB + lig * 16);
      Vec16<T>::unpack(vu, o);
      m = s_self;
      l = 1.f;
    }
  }

  bool ok = true;
  for (int t = 0; t < ntiles; ++t) {
    const int s = t % NSTAGE;
    if (ok && !mbar_wait_bounded(&bars[s], static_cast<uint32_t>((t / NSTAGE) & 1), kWaitLimit)) {
      ok = false;
      atomicOr(prm.err, ERR_MBAR_TIMEOUT);
    }
    const unsigned char* sK = stage_base + static_cast<size_t>(s) * Cfg::STAGE;
    const unsigned char* sV = sK + TILE * ROWB;
    const int rows = min(TILE, nrows - t * TILE);
    float lgi[IPW];
    int rowi[IPW];
#pragma unroll
    for (int i = 0; i < IPW; ++i) {
      const int row = warp * Cfg::RPW + i * RPI + grp;
      rowi[i] = row;
      float acc = 0.f;
      if (ok && row < rows) {
        float kf[EPV];
        Vec16<T>::unpack(*reinterpret_cast<const uint4*>(sK + row * ROWB + lig * 16), kf);
#pragma unroll
        for (int e = 0; e < EPV; ++e) acc = fmaf(qv[e], kf[e], acc);
      }
#pragma unroll
      for (int off = LPR / 2; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      lgi[i] = (ok && row < rows) ? acc : kNeg;
    }
    float mt = m;
#pragma unroll
    for (int i = 0; i < IPW; ++i) mt = fmaxf(mt, lgi[i]);
    const float corr = exp2f(m - mt);
    l *= corr;
#pragma unroll
    for (int e = 0; e < EPV; ++e) o[e] *= corr;
    m = mt;
#pragma unroll
    for (int i = 0; i < IPW; ++i) {
      if (ok && rowi[i] < rows) {
        const float w = exp2f(lgi[i] - m);
        l += w;
        float vf[EPV];
        Vec16<T>::unpack(*reinterpret_cast<const uint4*>(sV + rowi[i] * ROWB + lig * 16), vf);
#pragma unroll
        for (int e = 0; e < EPV; ++e) o[e] = fmaf(w, vf[e], o[e]);
        if (lig == 0) lg[t * TILE + rowi[i]] = lgi[i];
      }
    }
    __syncthreads();  // every warp is done with stage s
    if (tid == 0 && ok && t + NSTAGE < ntiles) {
      const int tn = t + NSTAGE;
      const int rn = min(TILE, nrows - tn * TILE);
      const uint32_t bytes = static_cast<uint32_t>(rn * ROWB);
      unsigned char* st = stage_base + static_cast<size_t>(s) * Cfg::STAGE;
      mbar_arrive_expect_tx(&bars[s], 2 * bytes);
      bulk_g2s_stream(st, gK + static_cast<size_t>(tn) * TILE * ROWB, bytes, &bars[s], policy);
      bulk_g2s_stream(st + TILE * ROWB, gV + static_cast<size_t>(tn) * TILE * ROWB, bytes, &bars[s], policy);
    }
  }
  griddep_launch();

  // merge the row groups of this warp (identical result in every lane group)
#pragma unroll
  for (int off = LPR; off < 32; off <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
    const float M = fmaxf(m, m2);
    const float a = exp2f(m - M), b = exp2f(m2 - M);
    l = l * a + l2 * b;
#pragma unroll
    for (int e = 0; e < EPV; ++e) o[e] = o[e] * a + __shfl_xor_sync(0xffffffffu, o[e], off) * b;
    m = M;
  }
  float* myred = red + warp * (D + 4);
  if (lane == 0) {
    myred[0] = m;
    myred[1] = l;
  }
  if (grp == 0) {
#pragma unroll
    for (int e = 0; e < EPV; ++e) myred[4 + lig * EPV + e] = o[e];
  }
  __syncthreads();
  if (tid < D) {
    float M = kNeg;
    for (int w = 0; w < Cfg::NW; ++w) M = fmaxf(M, red[w * (D + 4)]);
    float Ls = 0.f, Od = 0.f;
    for (int w = 0; w < Cfg::NW; ++w) {
      const float a = exp2f(red[w * (D + 4)] - M);
      Ls = fmaf(red[w * (D + 4) + 1], a, Ls);
      Od = fmaf(red[w * (D + 4) + 4 + tid], a, Od);
    }
    xo[tid] = Od;
    if (tid == 0) {
      xch->m = M;
      xch->l = Ls;
      xch->s_self = s_self;
    }
  }
  cluster.sync();  // (1) every CTA's partial softmax is published

  if (tid < S) {
    const Xch* rx = cluster.map_shared_rank(xch, tid);
    g_m[tid] = rx->m;
    g_l[tid] = rx->l;
    if (tid == 0) g_self[0] = rx->s_self;
  }
  __syncthreads();
  float M = kNeg;
  for (int r = 0; r < S; ++r) M = fmaxf(M, g_m[r]);
  float Ls = 0.f;
  for (int r = 0; r < S; ++r) Ls = fmaf(g_l[r], exp2f(g_m[r] - M), Ls);
  const float inv = 1.f / Ls;
  const float p_self = exp2f(g_self[0] - M) * inv;

  if (rank == 0 && tid < D) {
    float acc = 0.f;
    for (int r = 0; r < S; ++r) acc = fmaf(cluster.map_shared_rank(xo, r)[tid], exp2f(g_m[r] - M), acc);
    prm.out[static_cast<size_t>(pair) * D + tid] = acc * inv;
  }

  // probabilities -> accumulated scores; local minimum candidate key
  const int limit = p - R;  // candidates: kept positions <= p - R
  unsigned long long kmin = ~0ull;
  int smin = -1;
  for (int j = tid; j < nrows; j += NT) {
    const float ns = sc[j] + exp2f(lg[j] - M) * inv;
    sc[j] = ns;
    if (full && ps[j] <= limit) {
      const unsigned long long key =
          (static_cast<unsigned long long>(__float_as_uint(ns)) << 32) | static_cast<uint32_t>(ps[j]);
      if (key < kmin) {
        kmin = key;
        smin = lo + j;
      }
    }
  }
  unsigned long long wk = kmin;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const unsigned long long other = __shfl_xor_sync(0xffffffffu, wk, off);
    wk = other < wk ? other : wk;
  }
  if (lane == 0) blk_key[warp] = wk;
  __syncthreads();
  unsigned long long bk = blk_key[0];
  for (int w = 1; w < Cfg::NW; ++w) bk = blk_key[w] < bk ? blk_key[w] : bk;
  if (tid == 0) blk_slot = -1;
  __syncthreads();
  if (kmin == bk && kmin != ~0ull) blk_slot = smin;  // keys are unique (positions are)
  __syncthreads();
  if (tid == 0) {
    xch->key = bk;
    xch->slot = blk_slot;
  }
  cluster.sync();  // (2) every CTA's candidate is published

  int u;
  if (full) {
    if (tid < S) {
      const Xch* rx = cluster.map_shared_rank(xch, tid);
      g_key[tid] = rx->key;
      g_slot[tid] = rx->slot;
    }
    __syncthreads();
    unsigned long long best = ~0ull;
    u = -1;
    for (int r = 0; r < S; ++r)
      if (g_key[r] < best) {
        best = g_key[r];
        u = g_slot[r];
      }
    if (u < 0 && tid == 0) atomicOr(prm.err, ERR_NO_CANDIDATE);
  } else {
    u = count;
  }

  // write back: scores of this CTA's slots, the new token into slot u
  for (int j = tid; j < nrows; j += NT) prm.score[slot0 + j] = (lo + j == u) ? p_self : sc[j];
  if (u >= lo && u < lo + prm.chunk && u >= 0) {
    const size_t us = static_cast<size_t>(pair) * C + u;
    if (tid < 2 * LPR) {
      const int part = tid % LPR;
      const unsigned char* src = static_cast<const unsigned char*>(tid < LPR ? prm.k_new : prm.v_new) +
                                 static_cast<size_t>(pair) * ROWB + part * 16;
      unsigned char* dst = static_cast<unsigned char*>(tid < LPR ? prm.K : prm.V) + us * ROWB + part * 16;
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
    }
    if (tid == 0) {
      prm.pos[us] = p;
      if (u >= hi) prm.score[us] = p_self;  // fill phase: slot was empty
    }
  }
  if (rank == 0 && tid == 0) {
    if (u >= 0) prm.ring[static_cast<size_t>(pair) * R + head] = u;
    PairCtr nc;
    nc.p = p + 1;
    nc.count = full ? C : count + 1;
    nc.head = (head + 1) % R;
    nc.pad = 0;
    prm.ctr[pair] = nc;
    if (prm.evicted) prm.evicted[pair] = full ? u : -1;
  }
  cluster.sync();  // (3) no CTA leaves while its shared memory may be read
}

template <typename T, int D, int NT, int TILE, int NSTAGE>
cudaError_t launch_t(const DecodeParams& prm, int pairs, int splits, cudaStream_t s) {
  using Cfg = DecodeCfg<T, D, NT, TILE, NSTAGE>;
  using Lay = Layout<D, Cfg::NW, Cfg::STAGE, NSTAGE>;
  auto kern = decode_kernel<T, D, NT, TILE, NSTAGE>;
  const size_t smem = Lay::bytes(prm.chunk);
  // the limit is set for the largest chunk once, so later launches (also
  // inside graph capture) make no attribute calls
  cudaError_t e = kernel_attrs(reinterpret_cast<const void*>(kern), Lay::bytes(kMaxChunk), true);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(splits, pairs, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, prm);
}

constexpr int kThreads = 128;
constexpr int kTile = 16;
constexpr int kStages = 4;

}  // namespace

int decode_max_chunk() { return kMaxChunk; }

namespace {
template <typename T, int D>
cudaError_t feasible_t(int splits, int chunk, int pairs, int* clusters) {
  using Cfg = DecodeCfg<T, D, kThreads, kTile, kStages>;
  using Lay = Layout<D, Cfg::NW, Cfg::STAGE, kStages>;
  auto kern = decode_kernel<T, D, kThreads, kTile, kStages>;
  const size_t smem = Lay::bytes(chunk);
  cudaError_t e = kernel_attrs(reinterpret_cast<const void*>(kern), Lay::bytes(kMaxChunk), true);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(splits, pairs, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(clusters, kern, &cfg);
}
}  // namespace

// Number of clusters of `splits` CTAs the device can hold at once (0 = the
// cluster shape cannot be scheduled).
int decode_max_active_clusters(int dtype, int D, int splits, int chunk, int pairs) {
  int n = 0;
  cudaError_t e = cudaErrorInvalidValue;
  if (dtype == 0 && D == 128) e = feasible_t<__half, 128>(splits, chunk, pairs, &n);
  if (dtype == 0 && D == 64) e = feasible_t<__half, 64>(splits, chunk, pairs, &n);
  if (dtype == 1 && D == 128) e = feasible_t<float, 128>(splits, chunk, pairs, &n);
  if (dtype == 1 && D == 64) e = feasible_t<float, 64>(splits, chunk, pairs, &n);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_decode(const DecodeParams& prm, int dtype, int D, int pairs, int splits, int threads,
                          cudaStream_t s) {
  (void)threads;
  if (dtype == 0 && D == 128) return launch_t<__half, 128, kThreads, kTile, kStages>(prm, pairs, splits, s);
  if (dtype == 0 && D == 64) return launch_t<__half, 64, kThreads, kTile, kStages>(prm, pairs, splits, s);
  if (dtype == 1 && D == 128) return launch_t<float, 128, kThreads, kTile, kStages>(prm, pairs, splits, s);
  if (dtype == 1 && D == 64) return launch_t<float, 64, kThreads, kTile, kStages>(prm, pairs, splits, s);
  return cudaErrorInvalidValue;
}

}  // namespace h2o
