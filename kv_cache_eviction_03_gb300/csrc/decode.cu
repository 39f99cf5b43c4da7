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
// CTAs; CTA r owns the contiguous slot range [r*chunk, (r+1)*chunk), and S is
// chosen so that every CTA of the grid is resident at once.
//
// Inside a CTA one producer warp streams the CTA's K and V rows, 16 rows per
// stage, through a ring of shared-memory stages with 1-D bulk async copies
// (cp.async.bulk, full/empty mbarriers, L2 evict-first); four consumer warps
// compute the logits and a base-2 online softmax (m, l, o) per row group and
// release each stage with an mbarrier arrive, so the streaming loop has no
// block-wide barrier.  When the previous kernel on the stream worked on a
// different cache, the producer starts streaming before the programmatic
// grid-dependency wait, overlapping this step's loads with the tail of the
// previous kernel; only reads of the step's inputs (q, k_new, v_new) and all
// writes wait for it.
//
// The cluster's CTAs then exchange partial (m, l, o) through distributed
// shared memory, so every CTA knows the pair's global max and normaliser
// without a second pass over K: each turns its own logits (kept in shared
// memory) into probabilities, adds them to its slots' scores, and proposes its
// lowest candidate key (score bits, position) packed in 64 bits (non-negative
// float bits order like the floats).  The cluster minimum is the victim; the
// CTA that owns it writes the new row.  Cluster barriers are hardware barriers
// of co-scheduled CTAs: no CTA spins on another.
#include <cooperative_groups.h>
#include <cuda_fp16.h>

#include "h2o_internal.cuh"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace h2o {
namespace {

constexpr float kNeg = -3.0e38f;  // finite "minus infinity" for running maxima
// Every wait in this kernel is on work of this same grid (bulk copies it
// issued, stages its own warps release), so it completes within microseconds;
// 200k polls of <= 1 us each is a generous bound.
constexpr uint32_t kWaitLimit = 200000u;
constexpr int kMaxChunk = 4096;

template <typename T, int D, int NCW, int TILE>
struct DecodeCfg {
  static constexpr int E = sizeof(T);
  static constexpr int ROWB = D * E;     // bytes per K or V row
  static constexpr int EPV = 16 / E;     // elements per 16-byte vector
  static constexpr int LPR = ROWB / 16;  // lanes per row
  static constexpr int RPI = 32 / LPR;   // rows per warp-wide load
  static constexpr int NW = NCW + 1;     // consumer warps + one producer warp
  static constexpr int NT = NW * 32;
  static constexpr int STAGE = 2 * TILE * ROWB;
  static_assert(LPR >= 1 && LPR <= 32, "row must be 16..512 bytes");
  static_assert(TILE % RPI == 0, "a stage holds whole row groups");
  static_assert(NCW * 32 >= D, "one consumer thread per output dimension in the merge");
  static_assert(TILE <= 64, "per-warp weight buffer holds 64 rows");
};

constexpr int kMaxStages = 16;

struct __align__(16) Xch {
  float m, l, s_self, pad;
  unsigned long long key;
  int slot, pad2;
};

// Shared-memory layout (bytes); identical on host and device.  The stage ring
// depth and the CTA's slot count are launch parameters.
template <int D, int NCW, int STAGE>
struct Layout {
  static constexpr size_t full = 0;                            // kMaxStages mbarriers
  static constexpr size_t empty = 8 * kMaxStages;              // kMaxStages mbarriers
  static constexpr size_t xch = 16 * kMaxStages;
  static constexpr size_t xo = xch + sizeof(Xch);              // cluster-visible partial o[D]
  static constexpr size_t red = (xo + D * 4 + 127) / 128 * 128;
  static constexpr size_t gm = red + NCW * (D + 4) * 4;        // per-rank m / l / self / key / slot
  static constexpr size_t blk = gm + 16 * 24;                  // block argmin scratch + counters
  static constexpr size_t wbuf = (blk + 12 * (NCW + 1) + 16 + 15) / 16 * 16;  // per-warp row weights
  static constexpr size_t stages = (wbuf + NCW * 64 * 4 + 127) / 128 * 128;
  __host__ __device__ static size_t tail(int nstage) { return stages + static_cast<size_t>(nstage) * STAGE; }
  __host__ __device__ static size_t bytes(int nstage, int chunk) {
    return tail(nstage) + static_cast<size_t>(chunk) * 12;  // logits, scores, positions
  }
};

__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <typename T, int D, int NCW, int TILE>
__global__ void __launch_bounds__((NCW + 1) * 32, 4) decode_kernel(const DecodeParams prm) {
  using Cfg = DecodeCfg<T, D, NCW, TILE>;
  using Lay = Layout<D, NCW, Cfg::STAGE>;
  // Stage s is always consumed by warp s % NCW: with a ring depth that is a
  // multiple of NCW a warp never waits two phases ahead on a stage another
  // warp still owns, so mbarrier parity waits cannot alias.  Other depths
  // are rejected on the host; a kernel given one does no streaming.
  const int NSTAGE = prm.nstage;
  const bool ring_ok = NSTAGE >= NCW && NSTAGE % NCW == 0 && NSTAGE <= kMaxStages;
  constexpr int EPV = Cfg::EPV, LPR = Cfg::LPR, RPI = Cfg::RPI, ROWB = Cfg::ROWB;
  constexpr int NT = Cfg::NT, NW = Cfg::NW;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + Lay::full);
  uint64_t* empty_bar = reinterpret_cast<uint64_t*>(smem + Lay::empty);
  Xch* xch = reinterpret_cast<Xch*>(smem + Lay::xch);
  float* xo = reinterpret_cast<float*>(smem + Lay::xo);
  float* red = reinterpret_cast<float*>(smem + Lay::red);
  float* g_m = reinterpret_cast<float*>(smem + Lay::gm);
  float* g_l = g_m + 16;
  float* g_self = g_l + 16;
  unsigned long long* g_key = reinterpret_cast<unsigned long long*>(g_self + 16);
  int* g_slot = reinterpret_cast<int*>(g_key + 16);
  unsigned long long* blk_key = reinterpret_cast<unsigned long long*>(smem + Lay::blk);
  int* blk_slot = reinterpret_cast<int*>(blk_key + NW);  // per-warp candidate slot
  int* blk_int = blk_slot + NW;                           // [1..3] p, count, head
  float* wbuf = reinterpret_cast<float*>(smem + Lay::wbuf);
  unsigned char* stage_base = smem + Lay::stages;
  float* lg = reinterpret_cast<float*>(smem + Lay::tail(NSTAGE));
  float* sc = lg + prm.chunk;
  int* ps = reinterpret_cast<int*>(sc + prm.chunk);

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int S = static_cast<int>(cluster.num_blocks());
  const int pair = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = lane / LPR, lig = lane % LPR;
  const int C = prm.C, R = prm.R;
  const int lo = rank * prm.chunk;
  const size_t slot0 = static_cast<size_t>(pair) * C + lo;

  if (tid == 0) {
    if (!ring_ok) atomicOr(prm.err, ERR_RING_TIMEOUT);
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  float m = kNeg, l = 0.f, o[EPV];
#pragma unroll
  for (int e = 0; e < EPV; ++e) o[e] = 0.f;
  float s_self = 0.f;
  int p = 0, count = 0, head = 0;

  if (warp == NCW) {
    // ---------------------------------------------------------- producer warp
    if (lane == 0) {
      // The slot store is read before the grid-dependency wait only when the
      // previous kernel on this stream did not touch this cache.
      if (!prm.prefetch) griddep_wait();
      const int cnt = prm.ctr[pair].count;
      const int nrows = ring_ok ? max(min(lo + prm.chunk, cnt) - lo, 0) : 0;
      const int ntiles = (nrows + TILE - 1) / TILE;
      const unsigned char* gK = static_cast<const unsigned char*>(prm.K) + slot0 * ROWB;
      const unsigned char* gV = static_cast<const unsigned char*>(prm.V) + slot0 * ROWB;
      const uint64_t policy = policy_evict_first();
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % NSTAGE, k = t / NSTAGE;
        // stages are only released once the consumers are past the
        // grid-dependency wait, whose length depends on earlier kernels: wait
        // for the dependency here too before waiting on a stage
        if (k == 1 && s == 0 && prm.prefetch) griddep_wait();
        if (k > 0 && !mbar_wait_bounded(&empty_bar[s], static_cast<uint32_t>((k - 1) & 1), kWaitLimit)) {
          atomicOr(prm.err, ERR_RING_TIMEOUT);
          break;
        }
        const int rows = min(TILE, nrows - t * TILE);
        const uint32_t bytes = static_cast<uint32_t>(rows * ROWB);
        unsigned char* st = stage_base + static_cast<size_t>(s) * Cfg::STAGE;
        mbar_arrive_expect_tx(&full_bar[s], 2 * bytes);
        bulk_g2s_stream(st, gK + static_cast<size_t>(t) * TILE * ROWB, bytes, &full_bar[s], policy);
        bulk_g2s_stream(st + TILE * ROWB, gV + static_cast<size_t>(t) * TILE * ROWB, bytes, &full_bar[s], policy);
        issued = t + 1;
      }
      // no copy may still be landing in shared memory when the CTA exits: the
      // last phase of every stage used has completed (immediately true once
      // the consumers have read it)
      for (int t = max(issued - NSTAGE, 0); t < issued; ++t)
        if (!mbar_wait_bounded(&full_bar[t % NSTAGE], static_cast<uint32_t>((t / NSTAGE) & 1), kWaitLimit))
          atomicOr(prm.err, ERR_RING_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- consumer warps
    // Cache-owned state (counters, scores, positions) may be read before the
    // grid-dependency wait under the same rule as the producer's prefetch;
    // the step's inputs (q, k_new, v_new) only after it.
    int4 ctr = make_int4(0, 0, 0, 0);
    int nrows = 0;
    auto load_state = [&]() {
      ctr = *reinterpret_cast<const int4*>(prm.ctr + pair);  // {p, count, head, -}
      nrows = ring_ok ? max(min(lo + prm.chunk, ctr.y) - lo, 0) : 0;
      for (int j = tid; j < nrows; j += NCW * 32) {
        sc[j] = prm.score[slot0 + j];
        ps[j] = prm.pos[slot0 + j];
      }
    };
    if (prm.prefetch) load_state();
    griddep_wait();    // every earlier kernel on the stream has completed
    if (!prm.prefetch) load_state();
    p = ctr.x;
    count = ctr.y;
    head = ctr.z;
    const int ntiles = (nrows + TILE - 1) / TILE;
    if (tid == 0) {
      blk_int[1] = p;
      blk_int[2] = count;
      blk_int[3] = head;
    }
    float qv[EPV];
    Vec16<T>::unpack(*reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(prm.q) +
                                                     static_cast<size_t>(pair) * ROWB + lig * 16),
                     qv);
#pragma unroll
    for (int e = 0; e < EPV; ++e) qv[e] *= prm.qscale;  // exp2(logit) is the softmax numerator
    if (rank == 0 && warp == 0) {
      // the new token attends to itself: row group 0 of warp 0 starts from it
      float kf[EPV];
      Vec16<T>::unpack(*reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(prm.k_new) +
                                                       static_cast<size_t>(pair) * ROWB + lig * 16),
                       kf);
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < EPV; ++e) acc = fmaf(qv[e], kf[e], acc);
#pragma unroll
      for (int off = LPR / 2; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      s_self = acc;
      if (grp == 0) {
        Vec16<T>::unpack(*reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(prm.v_new) +
                                                         static_cast<size_t>(pair) * ROWB + lig * 16),
                         o);
        m = s_self;
        l = 1.f;
      }
    }
    // Each consumer warp takes whole stages in turn (warp w: stages w, w+NCW,
    // ...).  Within a stage, row group g of the warp (LPR lanes) owns RG rows;
    // every lane accumulates partial dot products of those rows over its 16
    // bytes of the row, a butterfly exchange sums them so that lane group
    // members end up holding whole-row logits (DUP copies of each), and the
    // probabilities go through shared memory to the lanes that weight V.
    constexpr int G = RPI;          // row groups per warp
    constexpr int RG = TILE / G;    // rows per group per stage
    constexpr int DUP = LPR / RG;   // lanes holding each row's total
    static_assert(RG >= 1 && RG <= LPR && LPR % RG == 0, "butterfly shape");
    float* wb = wbuf + warp * TILE;
    // Every earlier kernel has completed, so the next step may start its own
    // prefetch now; triggering only after this step's inputs are loaded keeps
    // those small loads ahead of the next step's bulk traffic.
    griddep_launch();
    bool ok = true;
    for (int t = warp; t < ntiles; t += NCW) {
      const int s = t % NSTAGE;
      if (ok && !mbar_wait_bounded(&full_bar[s], static_cast<uint32_t>((t / NSTAGE) & 1), kWaitLimit)) {
        ok = false;
        atomicOr(prm.err, ERR_MBAR_TIMEOUT);
      }
      const unsigned char* sK = stage_base + static_cast<size_t>(s) * Cfg::STAGE;
      const unsigned char* sV = sK + TILE * ROWB;
      const int rows = ok ? min(TILE, nrows - t * TILE) : 0;
      float acc[RG];
#pragma unroll
      for (int r = 0; r < RG; ++r) {
        const int row = grp * RG + r;
        float kf[EPV];
        Vec16<T>::unpack(*reinterpret_cast<const uint4*>(sK + row * ROWB + lig * 16), kf);
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < EPV; ++e) a = fmaf(qv[e], kf[e], a);
        acc[r] = row < rows ? a : 0.f;
      }
      // butterfly: halve the rows held per lane at each step
#pragma unroll
      for (int off = LPR / 2, n = RG; off >= 1; off >>= 1) {
        if (n > 1) {
          const int half = n / 2;
          const bool hi = (lig & off) != 0;
#pragma unroll
          for (int i = 0; i < half; ++i) {
            const float keep = hi ? acc[half + i] : acc[i];
            const float send = hi ? acc[i] : acc[half + i];
            acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
          }
          n = half;
        } else {
          acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], off);
        }
      }
      const int rown = grp * RG + lig / DUP;  // the row whose logit this lane holds
      const bool valid = rown < rows;
      const float x = valid ? acc[0] : kNeg;
      float mx = x;
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mn = fmaxf(m, mx);
      const float corr = exp2f(m - mn);
      m = mn;
      if (lig % DUP == 0) {
        wb[rown] = valid ? exp2f(x - mn) : 0.f;
        if (valid) lg[t * TILE + rown] = x;
      }
      __syncwarp();
      l *= corr;
#pragma unroll
      for (int e = 0; e < EPV; ++e) o[e] *= corr;
#pragma unroll
      for (int r = 0; r < RG; ++r) {
        const int row = grp * RG + r;
        if (row < rows) {
          const float w = wb[row];
          l += w;
          float vf[EPV];
          Vec16<T>::unpack(*reinterpret_cast<const uint4*>(sV + row * ROWB + lig * 16), vf);
#pragma unroll
          for (int e = 0; e < EPV; ++e) o[e] = fmaf(w, vf[e], o[e]);
        }
      }
      __syncwarp();  // wb is rewritten by the next stage
      // stage s may be refilled; after a timeout the stage is not released,
      // so no new copy can target memory an unfinished copy still writes
      if (lane == 0 && ok) mbar_arrive(&empty_bar[s]);
    }

    // merge the row groups of this warp (identical result in every group)
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
    consumer_sync(NCW * 32);
    if (tid < D) {
      float M = kNeg;
      for (int w = 0; w < NCW; ++w) M = fmaxf(M, red[w * (D + 4)]);
      float Ls = 0.f, Od = 0.f;
      for (int w = 0; w < NCW; ++w) {
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
  }
  // A pair handled by one CTA needs no cluster barrier or distributed shared
  // memory: plain block barriers and local shared memory do.
  const bool clustered = S > 1;
  if (clustered)
    cluster.sync();  // (1) every CTA's partial softmax is published
  else
    __syncthreads();

  if (tid < S) {
    const Xch* rx = clustered ? cluster.map_shared_rank(xch, tid) : xch;
    g_m[tid] = rx->m;
    g_l[tid] = rx->l;
    if (tid == 0) g_self[0] = rx->s_self;
  }
  __syncthreads();
  p = blk_int[1];
  count = blk_int[2];
  head = blk_int[3];
  const bool full = count >= C;
  const int nrows = max(min(lo + prm.chunk, count) - lo, 0);
  float M = kNeg;
  for (int r = 0; r < S; ++r) M = fmaxf(M, g_m[r]);
  float Ls = 0.f;
  for (int r = 0; r < S; ++r) Ls = fmaf(g_l[r], exp2f(g_m[r] - M), Ls);
  const float inv = 1.f / Ls;
  const float p_self = exp2f(g_self[0] - M) * inv;

  if (rank == 0 && tid < D) {
    float acc = 0.f;
    for (int r = 0; r < S; ++r)
      acc = fmaf((clustered ? cluster.map_shared_rank(xo, r) : xo)[tid], exp2f(g_m[r] - M), acc);
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
  // warp minimum, and the slot of the lane that holds it (keys are unique:
  // positions are)
  unsigned long long wk = kmin;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const unsigned long long other = __shfl_xor_sync(0xffffffffu, wk, off);
    wk = other < wk ? other : wk;
  }
  const unsigned holder = __ballot_sync(0xffffffffu, kmin == wk && kmin != ~0ull);
  const int wslot = __shfl_sync(0xffffffffu, smin, holder ? __ffs(holder) - 1 : 0);
  if (lane == 0) {
    blk_key[warp] = wk;
    blk_slot[warp] = holder ? wslot : -1;
  }
  __syncthreads();
  unsigned long long bk = ~0ull;
  int bslot = -1;
  for (int w = 0; w < NW; ++w)
    if (blk_key[w] < bk) {
      bk = blk_key[w];
      bslot = blk_slot[w];
    }

  int u;
  if (clustered) {
    if (tid == 0) {
      xch->key = bk;
      xch->slot = bslot;
    }
    cluster.sync();  // (2) every CTA's candidate is published
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
    } else {
      u = count;
    }
  } else {
    u = full ? bslot : count;
  }
  if (full && u < 0 && tid == 0) atomicOr(prm.err, ERR_NO_CANDIDATE);
  if (clustered) cluster_arrive_release();  // this CTA reads no more remote shared memory

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
      if (u >= lo + nrows) prm.score[us] = p_self;  // fill phase: slot was empty
    }
  }
  if (rank == 0 && tid == 0) {
    if (u >= 0) prm.ring[static_cast<size_t>(pair) * R + head] = u;
    *reinterpret_cast<int4*>(prm.ctr + pair) = make_int4(p + 1, full ? C : count + 1, (head + 1) % R, 0);
    if (prm.evicted) prm.evicted[pair] = full ? u : -1;
  }
  if (clustered) cluster_wait_acquire();  // (3) peers are done reading this CTA's shared memory
}

template <typename T, int D>
struct Kern {
  static constexpr int NCW = 4, TILE = 16;
  using Cfg = DecodeCfg<T, D, NCW, TILE>;
  using Lay = Layout<D, NCW, Cfg::STAGE>;
  static constexpr auto fn = decode_kernel<T, D, NCW, TILE>;

  static size_t smem(int nstage, int chunk) { return Lay::bytes(nstage, chunk); }

  static cudaError_t attrs() {
    // raised once for the largest configuration, so later launches (also
    // inside stream capture) make no attribute calls
    size_t most = Lay::bytes(kMaxStages, kMaxChunk);
    if (most > 227 * 1024) most = 227 * 1024;
    return kernel_attrs(reinterpret_cast<const void*>(fn), most, true);
  }

  static cudaError_t launch(const DecodeParams& prm, int pairs, int splits, cudaStream_t s) {
    cudaError_t e = attrs();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(splits, pairs, 1);
    cfg.blockDim = dim3(Cfg::NT, 1, 1);
    cfg.dynamicSmemBytes = smem(prm.nstage, prm.chunk);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = splits;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = splits > 1 ? 2 : 1;  // one CTA per pair: no cluster
    return cudaLaunchKernelEx(&cfg, fn, prm);
  }

  // CTAs that can be resident at once for this shape (0 = cannot launch)
  static int resident(int splits, int nstage, int chunk, int pairs, int sms) {
    if (attrs() != cudaSuccess) return 0;
    const size_t bytes = smem(nstage, chunk);
    if (bytes > 227 * 1024) return 0;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, Cfg::NT, bytes) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(splits, pairs, 1);
    cfg.blockDim = dim3(Cfg::NT, 1, 1);
    cfg.dynamicSmemBytes = bytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) != cudaSuccess) return 0;
    const long long by_sm = static_cast<long long>(per_sm) * sms;
    const long long by_cluster = static_cast<long long>(clusters) * splits;
    return static_cast<int>(by_sm < by_cluster ? by_sm : by_cluster);
  }
};

int chunk_for(int C, int splits) {
  const int ch = (C + splits - 1) / splits;
  return (ch + 3) / 4 * 4;
}

template <typename F>
auto dispatch(int dtype, int D, F&& f) -> decltype(f(Kern<__half, 128>{})) {
  if (dtype == 0 && D == 128) return f(Kern<__half, 128>{});
  if (dtype == 0 && D == 64) return f(Kern<__half, 64>{});
  if (dtype == 1 && D == 128) return f(Kern<float, 128>{});
  return f(Kern<float, 64>{});
}

}  // namespace

int decode_max_chunk() { return kMaxChunk; }

int decode_chunk(int C, int splits) { return chunk_for(C, splits); }

int decode_max_stages() { return kMaxStages; }
int decode_stage_multiple() { return Kern<__half, 128>::NCW; }

int device_sms() {
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return sms;
}

int decode_resident(int dtype, int D, int splits, int nstage, int chunk, int pairs) {
  const int sms = device_sms();
  const int r = dispatch(dtype, D, [&](auto k) { return decltype(k)::resident(splits, nstage, chunk, pairs, sms); });
  cudaGetLastError();
  return r;
}

// Default launch shape.  Consecutive decode steps of different layers
// overlap: the next kernel's CTAs start filling their rings while this one
// finishes, so one step should take about 1.7 CTAs per SM (the largest
// cluster size whose grid stays within that, each CTA keeping at least 32
// slots), with a 12-stage ring (three stages in flight per consumer warp)
// when two such CTAs fit on an SM.  Grids that need several waves anyway
// (many pairs) use 4-stage rings so that more CTAs are resident.
DecodeShape decode_pick_shape(int dtype, int D, int pairs, int C) {
  const int sms = device_sms();
  const long long target = sms > 0 ? (17LL * sms) / 10 : 256;
  DecodeShape sh;
  sh.splits = 1;
  for (int s = 16; s >= 2; s /= 2) {
    const int ch = chunk_for(C, s);
    if (ch < 32 || ch > kMaxChunk) continue;
    if (static_cast<long long>(pairs) * s <= target) {
      sh.splits = s;
      break;
    }
  }
  while (sh.splits < 16 && chunk_for(C, sh.splits) > kMaxChunk) sh.splits *= 2;
  const long long ctas = static_cast<long long>(pairs) * sh.splits;
  sh.stages = 4;
  if (ctas <= 2LL * sms) {
    const int ch = chunk_for(C, sh.splits);
    for (int st : {12, 8}) {
      const int res = decode_resident(dtype, D, sh.splits, st, ch, pairs);
      if (res >= 2 * sms || static_cast<long long>(res) >= ctas) {
        sh.stages = st;
        break;
      }
    }
  }
  return sh;
}

cudaError_t launch_decode(const DecodeParams& prm, int dtype, int D, int pairs, int splits, int threads,
                          cudaStream_t s) {
  (void)threads;
  if ((dtype != 0 && dtype != 1) || (D != 64 && D != 128)) return cudaErrorInvalidValue;
  return dispatch(dtype, D, [&](auto k) { return decltype(k)::launch(prm, pairs, splits, s); });
}

int decode_threads() { return 160; }

}  // namespace h2o
