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
// (cp.async.bulk, full/empty mbarriers, L2 evict-first); six consumer warps
// (four when a cluster shares the pair)
// compute the logits and a base-2 online softmax (m, l, o) per row group and
// release each stage with an mbarrier arrive, so the streaming loop has no
// block-wide barrier.  When the previous kernel on the stream worked on a
// different cache, the producer starts streaming before the programmatic
// grid-dependency wait, overlapping this step's loads with the tail of the
// previous kernel; only reads of the step's inputs (q, k_new, v_new) and all
// writes wait for it.
//
// The cluster's CTAs then exchange their partial (m, l) without a second
// pass over K: each pushes its pair into every peer's shared memory with
// st.async stores whose bytes complete a transaction count on the receiver's
// mbarrier (rank 0 also receives the other ranks' partial output rows), and
// each waits only until the bytes it expects have landed.  Every CTA then
// knows the pair's global max and normaliser, turns its own logits (kept in
// shared memory) into probabilities, adds them to its slots' scores, and
// pushes its lowest candidate key (score bits, position, packed in 64 bits:
// non-negative float bits order like the floats) to every peer the same way.
// The cluster minimum is the victim; the CTA that owns it writes the new row.
// No CTA reads another's shared memory and every CTA waits for all bytes
// pushed into it, so there is no cluster barrier after the one at entry that
// guarantees every peer has set up its mbarriers.  A pair handled by a single
// CTA uses plain block barriers and local shared memory instead.
//
// Many short pairs (thousands of pairs of up to 1024 slots) go to a second
// kernel, decode_warp_kernel, further down: one warp per pair, persistent.
#include <cooperative_groups.h>
#include <cuda_fp16.h>

#include <array>
#include <algorithm>
#include <map>
#include <vector>
#include <mutex>

#include "h2o_internal.cuh"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace h2o {
namespace {

constexpr float kNeg = -3.0e38f;  // finite "minus infinity" for running maxima

#ifdef H2O_DECODE_TIMELINE
// Profiling build: per-CTA time stamps (ns) of the last launches, written by
// thread 0 (consumer warp 0, lane 0) at: 0 entry, 1 grid dependency
// released, 2 step inputs loaded, 3 first stage landed, 4 every consumer past
// its loop, 5 pair's softmax normaliser known, 6 victim known, 7 exit.
__device__ unsigned long long g_decode_tl[kTimelineSlots][kTimelineMaxCtas][kTimelineStamps];
__device__ __forceinline__ void tl_stamp(const DecodeParams& prm, int i) {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)::"memory");
  const int cta = static_cast<int>(blockIdx.y * gridDim.x + blockIdx.x);
  if (cta < kTimelineMaxCtas) g_decode_tl[prm.tl_slot & (kTimelineSlots - 1)][cta][i] = t;
}
#define H2O_TL(i)                        \
  do {                                   \
    if (threadIdx.x == 0) tl_stamp(prm, i); \
  } while (0)
#else
#define H2O_TL(i) \
  do {            \
  } while (0)
#endif
// Every wait in this kernel is on work of this same grid (bulk copies it
// issued, stages its own warps release), so it completes within microseconds;
// 200k polls of <= 1 us each is a generous bound.
constexpr uint32_t kWaitLimit = 200000u;
constexpr int kMaxChunk = 4096;

// How a warp reads K/V rows of this type and width: each lane takes 16 bytes
// of a row, so LPR lanes cover a row and a warp-wide load covers RPI rows.
template <typename T, int D>
struct RowGeom {
  static constexpr int E = sizeof(T);
  static constexpr int ROWB = D * E;     // bytes per K or V row
  static constexpr int EPV = 16 / E;     // elements per 16-byte vector
  static constexpr int LPR = ROWB / 16;  // lanes per row
  static constexpr int RPI = 32 / LPR;   // rows per warp-wide load
  static_assert(LPR >= 1 && LPR <= 32, "row must be 16..512 bytes");
};

template <typename T, int D, int NCW, int TILE, int NP = 1>
struct DecodeCfg : RowGeom<T, D> {
  using G = RowGeom<T, D>;
  static constexpr int NW = NCW + NP;    // consumer warps + NP producer warps
  static constexpr int NT = NW * 32;
  static constexpr int STAGE = 2 * TILE * G::ROWB;
  static_assert(TILE % G::RPI == 0, "a stage holds whole row groups");
  static_assert(NCW * 32 >= D, "one consumer thread per output dimension in the merge");
  static_assert(TILE <= 64, "per-warp weight buffer holds 64 rows");
};

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One warp attends to one stage of `rows` (<= TILE) K/V rows: the logits
// q . k_r (q pre-scaled into the base-2 domain) are kept in lg[0..rows), and
// each row group's running softmax state (m, l, o) absorbs its rows.  Row group g
// of the warp (LPR lanes) owns RG rows; every lane accumulates partial dot
// products of those rows over its 16 bytes of the row, a butterfly exchange
// sums them so that lane-group members end up holding whole-row logits (DUP
// copies of each), and the probabilities go through the warp's shared buffer
// wb to the lanes that weight V.  After the call the warp no longer reads the
// stage.  With k_empty / v_full (position rolling) the stage's halves have
// barriers of their own: the K half is released on k_empty as soon as the
// logits are formed, and the V half is waited for (v_full, phase parity
// v_par) only before the V rows are weighted; false if that wait gave up
// (the V rows are then not read).
// Position rolling: rotate this lane's EPV/2 element pairs (2i, 2i+1) of a
// row by r * theta_i, as in the rotary embedding, composed from the rank's
// digits: the rotation-table entry of level l's digit (rope_entry) holds
// cos and sin of the digit's angle for every pair, in shared memory in lane
// order: float4 h * LPR + lig of an entry holds, for this lane's pairs 2h and
// 2h + 1, (cos, cos, sin, sin), so that two pairs rotate in packed f32x2
// arithmetic.
template <int EPV, int D, int LPR>
__device__ __forceinline__ void rope_rotate_level(float (&x)[EPV], const float2* tab, int entry, int lig) {
  const float4* t = reinterpret_cast<const float4*>(tab + entry * (D / 2)) + lig;
#pragma unroll
  for (int h = 0; h < EPV / 4; ++h) {
    const float4 c = t[h * LPR];  // cos, cos, sin, sin of two pairs
    const float a0 = x[4 * h], a1 = x[4 * h + 1], b0 = x[4 * h + 2], b1 = x[4 * h + 3];
    x[4 * h] = a0 * c.x - a1 * c.z;
    x[4 * h + 1] = a0 * c.z + a1 * c.x;
    x[4 * h + 2] = b0 * c.y - b1 * c.w;
    x[4 * h + 3] = b0 * c.w + b1 * c.y;
  }
}
template <int EPV, int D, int LPR>
__device__ __forceinline__ void rope_rotate_digits(float (&x)[EPV], const float2* tab, int r, int levels, int low,
                                                   int hi, int lig) {
#pragma unroll
  for (int lv = 0; lv < 6; ++lv)
    if (lv < levels) rope_rotate_level<EPV, D, LPR>(x, tab, rope_entry(r, lv, low, hi), lig);
}
// The same rotation on a key held as real parts re[h] = (x[4h], x[4h+2]) and
// imaginary parts im[h] = (x[4h+1], x[4h+3]) of its pairs, two pairs per
// f32x2 instruction (each lane of an f32x2 operation rounds as the scalar
// fp32 operation would).
template <int NH, int D, int LPR>
__device__ __forceinline__ void rope_rotate_level2(float2 (&re)[NH], float2 (&im)[NH], const float2* tab, int entry,
                                                   int lig) {
  const float4* t = reinterpret_cast<const float4*>(tab + entry * (D / 2)) + lig;
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    const float4 c = t[h * LPR];
    const float2 cs = make_float2(c.x, c.y), sn = make_float2(c.z, c.w);
    const float2 rc = mul_f32x2(re[h], cs), rs = mul_f32x2(re[h], sn);
    const float2 nim = mul_f32x2(im[h], make_float2(-1.f, -1.f));
    re[h] = fma_f32x2(nim, sn, rc);    // re cos - im sin
    im[h] = fma_f32x2(im[h], cs, rs);  // re sin + im cos
  }
}

// Position rolling (ROPE): the logit of a key at rank r is
// Re sum_i conj(Q_i) T0[lowest digit of r]_i K'_i over the lane's pairs as complex
// numbers, Q the rotated query, T0 the level-0 table and K' the key rotated
// by the rank's higher digits (KL levels): tab's level-0 entries then hold
// P0[d] = conj(Q) T0[d], built once per step, so a key takes KL rotations.
// P0 is stored per two pairs as (Re, Re, -Im, -Im), and the rotations, the
// P0 dot product and the V accumulation run in f32x2.
template <typename T, int D, int TILE, bool ROPE = false, int KL = 0>
__device__ __forceinline__ bool attend_tile(const unsigned char* sK, const unsigned char* sV, int rows,
                                            const float (&qv)[RowGeom<T, D>::EPV], float& m, float& l,
                                            float (&o)[RowGeom<T, D>::EPV], float* wb, float* lg, int lane,
                                            const int* rk = nullptr, const float2* tab = nullptr, int low = 4,
                                            int hi = 4, uint64_t* k_empty = nullptr, uint64_t* v_full = nullptr,
                                            uint32_t v_par = 0) {
  using Gm = RowGeom<T, D>;
  constexpr int EPV = Gm::EPV, LPR = Gm::LPR, ROWB = Gm::ROWB;
  constexpr int G = Gm::RPI;      // row groups per warp
  constexpr int RG = TILE / G;    // rows per group per stage
  constexpr int DUP = LPR / RG;   // lanes holding each row's total
  static_assert(RG >= 1 && RG <= LPR && LPR % RG == 0, "butterfly shape");
  static_assert(!ROPE || EPV % 4 == 0, "a lane holds whole pairs of pairs");
  const int grp = lane / LPR, lig = lane % LPR;
  float acc[RG];
#pragma unroll
  for (int r = 0; r < RG; ++r) {
    const int row = grp * RG + r;
    float kf[EPV];
    Vec16<T>::unpack(*reinterpret_cast<const uint4*>(sK + row * ROWB + lig * 16), kf);
    float a = 0.f;
    if constexpr (ROPE) {  // key rotated to its rank inside the cache (rk: this stage's ranks)
      const int rr = row < rows ? rk[row] : 0;
      constexpr int NH = EPV / 4;
      float2 re[NH], im[NH];
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        re[h] = make_float2(kf[4 * h], kf[4 * h + 2]);
        im[h] = make_float2(kf[4 * h + 1], kf[4 * h + 3]);
      }
#pragma unroll
      for (int lv = 1; lv <= KL; ++lv)
        rope_rotate_level2<NH, D, LPR>(re, im, tab, rope_entry(rr, lv, low, hi), lig);
      const float4* z = reinterpret_cast<const float4*>(tab + rope_entry(rr, 0, low, hi) * (D / 2)) + lig;  // P0[d0]
      float2 a2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        const float4 c = z[h * LPR];
        a2 = fma_f32x2(re[h], make_float2(c.x, c.y), a2);
        a2 = fma_f32x2(im[h], make_float2(c.z, c.w), a2);
      }
      a = a2.x + a2.y;
    } else {
#pragma unroll
      for (int e = 0; e < EPV; ++e) a = fmaf(qv[e], kf[e], a);
    }
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
  // every lane's K reads are complete (their sums went through the exchange)
  if (k_empty != nullptr) {
    __syncwarp();
    if (lane == 0 && rows > 0) mbar_arrive(k_empty);
  }
  const int rown = grp * RG + lig / DUP;  // the row whose logit this lane holds
  const bool valid = rown < rows;
  const float x = valid ? acc[0] : kNeg;
  // running maximum per row group (its lanes weight only its own rows; the
  // groups' states are merged after the loop)
  float mx = x;
#pragma unroll
  for (int off = LPR / 2; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  const float mn = fmaxf(m, mx);
  const float corr = exp2f(m - mn);
  m = mn;
  if (lig % DUP == 0) {
    wb[rown] = valid ? exp2f(x - mn) : 0.f;
    if (valid) lg[rown] = x;
  }
  __syncwarp();
  l *= corr;
  if constexpr (ROPE) {
#pragma unroll
    for (int e = 0; e < EPV; e += 2) {
      const float2 oc = mul_f32x2(make_float2(o[e], o[e + 1]), make_float2(corr, corr));
      o[e] = oc.x;
      o[e + 1] = oc.y;
    }
  } else {
#pragma unroll
    for (int e = 0; e < EPV; ++e) o[e] *= corr;
  }
  int vrows = rows;
  bool v_ok = true;
  if (v_full != nullptr && rows > 0 && !mbar_wait_bounded(v_full, v_par, kWaitLimit)) {
    v_ok = false;
    vrows = 0;
  }
#pragma unroll
  for (int r = 0; r < RG; ++r) {
    const int row = grp * RG + r;
    if (row < vrows) {
      const float w = wb[row];
      l += w;
      float vf[EPV];
      Vec16<T>::unpack(*reinterpret_cast<const uint4*>(sV + row * ROWB + lig * 16), vf);
      if constexpr (ROPE) {
#pragma unroll
        for (int e = 0; e < EPV; e += 2) {
          const float2 oe = fma_f32x2(make_float2(w, w), make_float2(vf[e], vf[e + 1]), make_float2(o[e], o[e + 1]));
          o[e] = oe.x;
          o[e + 1] = oe.y;
        }
      } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e) o[e] = fmaf(w, vf[e], o[e]);
      }
    }
  }
  __syncwarp();  // wb is rewritten by the next stage
  return v_ok;
}

// Minimum over the warp of a 64-bit key (score bits << 32 | position), in
// two 32-bit warp reductions: the high words, then the low words of the
// lanes that hold the lowest high word.
__device__ __forceinline__ unsigned long long warp_min_key(unsigned long long key) {
  const unsigned hi = static_cast<unsigned>(key >> 32);
  const unsigned mh = __reduce_min_sync(0xffffffffu, hi);
  const unsigned ml = __reduce_min_sync(0xffffffffu, hi == mh ? static_cast<unsigned>(key) : 0xffffffffu);
  return (static_cast<unsigned long long>(mh) << 32) | ml;
}

// Merge the row groups of a warp: afterwards every group holds the same
// (m, l, o) over all rows the warp has seen.
template <typename T, int D>
__device__ __forceinline__ void merge_groups(float& m, float& l, float (&o)[RowGeom<T, D>::EPV]) {
  constexpr int EPV = RowGeom<T, D>::EPV, LPR = RowGeom<T, D>::LPR;
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
}

constexpr int kMaxStages = 18;
// Consumer warps of the cluster kernel.  A pair handled by one CTA gets six
// (two stages of the 12-stage ring in flight per warp), the CTAs of a
// cluster four (three each): measured, six is 2.5% faster than four for one
// CTA per pair (OPT-6.7B shape) and four is 1-3% faster in 2- and 8-CTA
// clusters (streaming, LLaMA-16K shapes).  With position rolling the loop is
// bound by the latency of each key's rotation, not by memory, and eight warps
// (one stage each of an 8-stage ring) hide it best: measured 12-17% faster
// than six or four on those three shapes; ten were no faster, and twelve
// no longer fit two CTAs on an SM.
__host__ __device__ constexpr int consumer_warps(int splits, bool rope = false) {
  return rope ? 8 : (splits > 1 ? 4 : 6);
}
// Producer warps: two (K rows and V rows under barriers of their own) where
// the stage halves are released separately, else one.  Measured: separate
// halves take the rolling kernel 4-7% faster (its logits are slow, and the K
// half refills meanwhile) and the plain kernel 9-17% slower, so only
// position rolling uses them.
__host__ __device__ constexpr bool split_halves(bool rope) { return rope; }
__host__ __device__ constexpr int producer_warps(bool rope) { return split_halves(rope) ? 2 : 1; }

// A CTA's merged partial softmax (max, normaliser, self logit).
struct __align__(16) Xch {
  float m, l, s_self, pad;
};

// Shared-memory layout (bytes); identical on host and device.  The stage ring
// depth, the CTA's slot count and the cluster size are launch parameters.
template <int D, int NCW, int TILE, int STAGE, bool ROPE>
struct Layout {
  static constexpr int PER_SLOT = ROPE ? 16 : 12;  // logit, score, position (, rank)
  static constexpr size_t full = 0;                            // kMaxStages mbarriers (K and V, or K)
  static constexpr size_t empty = 8 * kMaxStages;              // kMaxStages mbarriers (K and V, or K)
  static constexpr size_t fullv = 16 * kMaxStages;             // kMaxStages mbarriers (V, rolling)
  static constexpr size_t emptyv = 24 * kMaxStages;            // kMaxStages mbarriers (V, rolling)
  static constexpr size_t xbar = 32 * kMaxStages;              // mbarrier: the peers' partials have landed
  static constexpr size_t kbar = xbar + 8;                     // mbarrier: the peers' candidates have landed
  static constexpr size_t tbar = xbar + 16;                    // mbarrier: the rotation tables have landed
  static constexpr size_t xch = xbar + 32;
  static constexpr size_t xo = xch + sizeof(Xch);              // this CTA's partial o[D]
  static constexpr size_t gm = (xo + D * 4 + 15) / 16 * 16;    // per-rank partials [16], candidates [16]
  static constexpr size_t blk = gm + 16 * 32;                  // block argmin scratch + counters
  static constexpr size_t wbuf = (blk + 12 * (NCW + 2) + 16 + 15) / 16 * 16;  // per-warp row weights
  static constexpr size_t stages = (wbuf + NCW * TILE * 4 + 127) / 128 * 128;
  __host__ __device__ static size_t tail(int nstage) { return stages + static_cast<size_t>(nstage) * STAGE; }
  // after the logits, scores and positions of the CTA's slots: rank 0's
  // copies of the other ranks' partial output rows (rank r at r - 1)
  __host__ __device__ static size_t rows_in(int nstage, int chunk) {
    return (tail(nstage) + static_cast<size_t>(chunk) * PER_SLOT + 15) / 16 * 16;
  }
  // after the peers' rows: position rolling's rotation tables
  __host__ __device__ static size_t tab(int nstage, int chunk, int splits) {
    return (rows_in(nstage, chunk) + (splits > 1 ? static_cast<size_t>(splits - 1) * D * 4 : 0) + 15) / 16 * 16;
  }
  __host__ __device__ static size_t tab_bytes(int entries) {
    return ROPE ? static_cast<size_t>(entries) * (D / 2) * sizeof(float2) : 0;
  }
  __host__ __device__ static size_t bytes(int nstage, int chunk, int splits, int entries) {
    return tab(nstage, chunk, splits) + tab_bytes(entries);
  }
};

__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <typename T, int D, int NCW, int TILE, bool ROPE>
__global__ void __launch_bounds__((NCW + producer_warps(ROPE)) * 32, NCW > 6 ? 2 : (NCW > 4 ? 3 : 4))
    decode_kernel(const DecodeParams prm) {
  constexpr bool SPLIT = split_halves(ROPE);
  using Cfg = DecodeCfg<T, D, NCW, TILE, producer_warps(ROPE)>;
  using Lay = Layout<D, NCW, TILE, Cfg::STAGE, ROPE>;
  // Stage s is always consumed by warp s % NCW: with a ring depth that is a
  // multiple of NCW a warp never waits two phases ahead on a stage another
  // warp still owns, so mbarrier parity waits cannot alias.  Other depths
  // are rejected on the host; a kernel given one only reports it.
  const int NSTAGE = prm.nstage;
  if (!(NSTAGE >= NCW && NSTAGE % NCW == 0 && NSTAGE <= kMaxStages)) {
    if (threadIdx.x == 0) atomicOr(prm.err, ERR_RING_TIMEOUT);
    return;
  }
  constexpr int EPV = Cfg::EPV, LPR = Cfg::LPR, ROWB = Cfg::ROWB;
  constexpr int NT = Cfg::NT, NW = Cfg::NW;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + Lay::full);
  uint64_t* empty_bar = reinterpret_cast<uint64_t*>(smem + Lay::empty);
  uint64_t* fullv_bar = reinterpret_cast<uint64_t*>(smem + Lay::fullv);
  uint64_t* emptyv_bar = reinterpret_cast<uint64_t*>(smem + Lay::emptyv);
  Xch* xch = reinterpret_cast<Xch*>(smem + Lay::xch);
  float* xo = reinterpret_cast<float*>(smem + Lay::xo);
  Xch* xin = reinterpret_cast<Xch*>(smem + Lay::gm);         // rank r's (m, l, self) at [r]
  uint4* kin = reinterpret_cast<uint4*>(smem + Lay::gm + 256);  // rank r's candidate (key, slot) at [r]
  uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + Lay::xbar);
  uint64_t* kbar = reinterpret_cast<uint64_t*>(smem + Lay::kbar);
  uint64_t* tbar = reinterpret_cast<uint64_t*>(smem + Lay::tbar);
  unsigned long long* blk_key = reinterpret_cast<unsigned long long*>(smem + Lay::blk);
  int* blk_slot = reinterpret_cast<int*>(blk_key + NW);  // per-warp candidate slot
  int* blk_int = blk_slot + NW;                           // [1..3] p, count, head
  float* wbuf = reinterpret_cast<float*>(smem + Lay::wbuf);
  unsigned char* stage_base = smem + Lay::stages;
  float* lg = reinterpret_cast<float*>(smem + Lay::tail(NSTAGE));
  float* sc = lg + prm.chunk;
  int* ps = reinterpret_cast<int*>(sc + prm.chunk);
  int* rk = ps + prm.chunk;  // slot ranks inside the cache (position rolling only)
  float* xo_in = reinterpret_cast<float*>(smem + Lay::rows_in(NSTAGE, prm.chunk));

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int S = static_cast<int>(cluster.num_blocks());
  float2* rtab = reinterpret_cast<float2*>(smem + Lay::tab(NSTAGE, prm.chunk, S));  // rotation tables (rolling)
  const int pair = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = lane / LPR, lig = lane % LPR;
  const int C = prm.C, R = prm.R;
  const int lo = rank * prm.chunk;
  const size_t slot0 = static_cast<size_t>(pair) * C + lo;
  H2O_TL(0);

  if (tid == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
      if constexpr (SPLIT) {
        mbar_init(&fullv_bar[s], 1);
        mbar_init(&emptyv_bar[s], 1);
      }
    }
    mbar_init(xbar, 1);
    mbar_init(kbar, 1);
    mbar_init(tbar, 1);
    fence_mbar_init();
    if (S > 1) {
      // the bytes the peers will push: (m, l, self) from each, the partial
      // output rows into rank 0, and later one candidate from each
      mbar_arrive_expect_tx(xbar, static_cast<uint32_t>((S - 1) * 16 + (rank == 0 ? (S - 1) * D * 4 : 0)));
      mbar_arrive_expect_tx(kbar, static_cast<uint32_t>((S - 1) * 16));
    }
  }
  __syncthreads();
  // The cluster's CTAs exchange partial results by writing into each other's
  // shared memory; this arrival (waited for before the first such write)
  // guarantees every peer has started.
  if (S > 1) cluster_arrive_relaxed();

  float m = kNeg, l = 0.f, o[EPV];
#pragma unroll
  for (int e = 0; e < EPV; ++e) o[e] = 0.f;
  float s_self = 0.f;
  int p = 0, count = 0, head = 0;
  uint4 newrow = make_uint4(0, 0, 0, 0);

  if (warp >= NCW) {
    // -------------------------------------------------------- producer warp(s)
    // One warp copies each tile's K and V rows into its stage under one pair
    // of barriers (full_bar / empty_bar).  With position rolling, where a
    // tile's logits take much longer than its memory, warp NCW copies the K
    // rows (full_bar / empty_bar) and warp NCW + 1 the V rows (fullv_bar /
    // emptyv_bar): the K half of a stage is refilled while its consumer still
    // weights the V half.
    const int part = SPLIT ? warp - NCW : 2;  // 0: K rows, 1: V rows, 2: both
    if (lane == 0) {
      uint64_t* fb = part == 1 ? fullv_bar : full_bar;
      uint64_t* eb = part == 1 ? emptyv_bar : empty_bar;
      // position rolling: the rotation tables, constant while rolling is on,
      // so they are copied before any wait
      const uint32_t tbytes =
          static_cast<uint32_t>(Lay::tab_bytes(rope_entries_for(C, prm.rope_low_bits, prm.rope_hi_bits)));
      if constexpr (ROPE) {
        if (part == 0) {
          mbar_arrive_expect_tx(tbar, tbytes);
          bulk_g2s(rtab, prm.rope, tbytes, tbar);
        }
      }
      // The slot store is read before the grid-dependency wait only when the
      // previous kernel on this stream did not touch this cache.  Then the
      // first tile of the CTA's slot range is requested at once, before the
      // pair's count is known (a full cache uses it; rows past the count are
      // never read), so the first stage does not wait for that load.  The
      // rest follows the count: a whole ring requested that early would put
      // the consumers' small loads behind megabytes of bulk reads.
      const unsigned char* gK = static_cast<const unsigned char*>(prm.K) + slot0 * ROWB;
      const unsigned char* gV = static_cast<const unsigned char*>(prm.V) + slot0 * ROWB;
      const uint64_t policy = policy_evict_first();
      auto issue = [&](int t, int s, int rows) {
        const uint32_t bytes = static_cast<uint32_t>(rows * ROWB);
        unsigned char* st = stage_base + static_cast<size_t>(s) * Cfg::STAGE;
        const size_t off = static_cast<size_t>(t) * TILE * ROWB;
        mbar_arrive_expect_tx(&fb[s], part == 2 ? 2 * bytes : bytes);
        if (part != 1) bulk_g2s_stream(st, gK + off, bytes, &fb[s], policy);
        if (part != 0) bulk_g2s_stream(st + TILE * ROWB, gV + off, bytes, &fb[s], policy);
      };
      int issued = 0;
      if (prm.prefetch) {
        const int rows0 = min(TILE, max(min(lo + prm.chunk, C) - lo, 0));  // inside the pair's slots
        if (rows0 > 0) {
          issue(0, 0, rows0);
          issued = 1;
        }
      } else {
        griddep_wait();
      }
      const int cnt = prm.ctr[pair].count;
      const int nrows = max(min(lo + prm.chunk, cnt) - lo, 0);
      const int ntiles = (nrows + TILE - 1) / TILE;
      for (int t = issued; t < ntiles; ++t) {
        const int s = t % NSTAGE, k = t / NSTAGE;
        // stages are only released once the consumers are past the
        // grid-dependency wait, whose length depends on earlier kernels: wait
        // for the dependency here too before waiting on a stage
        if (k == 1 && s == 0 && prm.prefetch) griddep_wait();
        if (k > 0 && !mbar_wait_bounded(&eb[s], static_cast<uint32_t>((k - 1) & 1), kWaitLimit)) {
          atomicOr(prm.err, ERR_RING_TIMEOUT);
          break;
        }
        issue(t, s, min(TILE, nrows - t * TILE));
        issued = t + 1;
      }
      // no copy may still be landing in shared memory when the CTA exits: the
      // last phase of every stage used has completed (immediately true once
      // the consumers have read it)
      for (int t = max(issued - NSTAGE, 0); t < issued; ++t)
        if (!mbar_wait_bounded(&fb[t % NSTAGE], static_cast<uint32_t>((t / NSTAGE) & 1), kWaitLimit))
          atomicOr(prm.err, ERR_RING_TIMEOUT);
      if constexpr (ROPE)
        if (part == 0 && !mbar_wait_bounded(tbar, 0u, kWaitLimit)) atomicOr(prm.err, ERR_RING_TIMEOUT);
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
      // The scores and positions are needed only in the epilogue, the ranks
      // (position rolling) from the loop on: they come by asynchronous copies
      // over the CTA's whole slot range (no wait for the count first), so no
      // consumer stalls on them before the grid-dependency wait; each thread
      // completes its own copies before the first use.
      const int cap = max(min(lo + prm.chunk, C) - lo, 0);
      for (int j = tid; j < cap; j += NCW * 32) {
        cp_async4(sc + j, prm.score + slot0 + j);
        cp_async4(ps + j, prm.pos + slot0 + j);
        if constexpr (ROPE) cp_async4(rk + j, prm.rank + slot0 + j);
      }
      cp_async_commit();
      ctr = *reinterpret_cast<const int4*>(prm.ctr + pair);  // {p, count, head, -}
      nrows = max(min(lo + prm.chunk, ctr.y) - lo, 0);
    };
    // warm L2 with this pair's q, k_new and v_new rows while waiting
    {
      constexpr int NLINE = (ROWB + 127) / 128;
      if (tid < 3 * NLINE) {
        const void* row = tid < NLINE ? prm.q : (tid < 2 * NLINE ? prm.k_new : prm.v_new);
        prefetch_l2(static_cast<const unsigned char*>(row) + static_cast<size_t>(pair) * ROWB + (tid % NLINE) * 128);
      }
    }
    if (prm.prefetch) load_state();
    griddep_wait();    // every earlier kernel on the stream has completed
    H2O_TL(1);
    if (!prm.prefetch) load_state();
    // the slice of the new K (threads < LPR) or V row (LPR..2 LPR-1) that
    // this thread writes if this CTA owns the evicted slot
    if (tid < 2 * LPR)
      newrow = *reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(tid < LPR ? prm.k_new : prm.v_new) +
                                               static_cast<size_t>(pair) * ROWB + (tid % LPR) * 16);
    p = ctr.x;
    count = ctr.y;
    head = ctr.z;
    const int ntiles = (nrows + TILE - 1) / TILE;
    if (tid == 0) {
      blk_int[1] = p;
      blk_int[2] = count;
      blk_int[3] = head;
    }
    // q, and for the self term k_new and v_new, requested together (one
    // round trip rather than three)
    const size_t in_off = static_cast<size_t>(pair) * ROWB + lig * 16;
    const uint4 q4 = *reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(prm.q) + in_off);
    uint4 k4 = make_uint4(0, 0, 0, 0), v4 = make_uint4(0, 0, 0, 0);
    if (rank == 0 && warp == 0) {
      k4 = *reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(prm.k_new) + in_off);
      v4 = *reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(prm.v_new) + in_off);
    }
    float qv[EPV];
    Vec16<T>::unpack(q4, qv);
#pragma unroll
    for (int e = 0; e < EPV; ++e) qv[e] *= prm.qscale;  // exp2(logit) is the softmax numerator
    H2O_TL(2);
    // position rolling: the query (and the new key) sit at rank `count`, after
    // every kept token
    if constexpr (ROPE) {
      if (!mbar_wait_bounded(tbar, 0u, kWaitLimit)) atomicOr(prm.err, ERR_MBAR_TIMEOUT);
      rope_rotate_digits<EPV, D, LPR>(qv, rtab, count, prm.rope_levels, prm.rope_low_bits, prm.rope_hi_bits, lig);
    }
    if (rank == 0 && warp == 0) {
      // the new token attends to itself: row group 0 of warp 0 starts from it
      float kf[EPV];
      Vec16<T>::unpack(k4, kf);
      if constexpr (ROPE)
        rope_rotate_digits<EPV, D, LPR>(kf, rtab, count, prm.rope_levels, prm.rope_low_bits, prm.rope_hi_bits, lig);
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < EPV; ++e) acc = fmaf(qv[e], kf[e], acc);
#pragma unroll
      for (int off = LPR / 2; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      s_self = acc;
      if (grp == 0) {
        Vec16<T>::unpack(v4, o);
        m = s_self;
        l = 1.f;
      }
    }
    // Each consumer warp takes whole stages in turn (warp w: stages w, w+NCW,
    // ...).
    float* wb = wbuf + warp * TILE;
    // Every earlier kernel has completed, so the next step may start its own
    // prefetch now; triggering only after this step's inputs are loaded keeps
    // those small loads ahead of the next step's bulk traffic.
    griddep_launch();
    if constexpr (ROPE) {
      // after the barrier every rank in rk[] is in place, and every read of
      // the level-0 table (query, new key) is done: the level-0 entries become
      // P0[d] = conj(Q) T0[d], digit d built by row group (warp * G + grp)
      // when d is congruent to it modulo the consumers' row groups
      cp_async_wait<0>();
      consumer_sync(NCW * 32);
      constexpr int NG = NCW * Cfg::RPI;
      const int n0 = prm.rope_levels > 1 ? 1 << prm.rope_low_bits : C + 1;  // level-0 entries
      for (int d = warp * Cfg::RPI + grp; d < n0; d += NG) {
        float4* e = reinterpret_cast<float4*>(rtab + d * (D / 2)) + lig;
#pragma unroll
        for (int h = 0; h < EPV / 4; ++h) {
          const float4 c = e[h * LPR];  // cos, cos, sin, sin of pairs 2h, 2h + 1
          const float qa = qv[4 * h], qb = qv[4 * h + 1], qc = qv[4 * h + 2], qd = qv[4 * h + 3];
          // conj(qa + i qb) (cos + i sin) and conj(qc + i qd) (cos + i sin):
          // real parts, then negated imaginary parts
          e[h * LPR] = make_float4(qa * c.x + qb * c.z, qc * c.y + qd * c.w, qb * c.x - qa * c.z, qd * c.y - qc * c.w);
        }
      }
      consumer_sync(NCW * 32);
    }
    bool ok = true;
    for (int t = warp; t < ntiles; t += NCW) {
      const int s = t % NSTAGE;
      if (ok && !mbar_wait_bounded(&full_bar[s], static_cast<uint32_t>((t / NSTAGE) & 1), kWaitLimit)) {
        ok = false;
        atomicOr(prm.err, ERR_MBAR_TIMEOUT);
      }
      if (t == 0) H2O_TL(3);
      const unsigned char* sK = stage_base + static_cast<size_t>(s) * Cfg::STAGE;
      const int rows = ok ? min(TILE, nrows - t * TILE) : 0;
      if constexpr (ROPE) {
        const int* rks = rk + t * TILE;
        float* lgs = lg + t * TILE;
        const int low = prm.rope_low_bits, hi = prm.rope_hi_bits;
        uint64_t* ke = &empty_bar[s];  // the K half goes back inside attend_tile
        uint64_t* vf = &fullv_bar[s];
        const uint32_t par = static_cast<uint32_t>((t / NSTAGE) & 1);
        bool v_ok = true;
        switch (prm.rope_levels) {  // key-side rotations: the digits above the lowest
          case 1: v_ok = attend_tile<T, D, TILE, true, 0>(sK, sK + TILE * ROWB, rows, qv, m, l, o, wb, lgs, lane, rks, rtab, low, hi, ke, vf, par); break;
          case 2: v_ok = attend_tile<T, D, TILE, true, 1>(sK, sK + TILE * ROWB, rows, qv, m, l, o, wb, lgs, lane, rks, rtab, low, hi, ke, vf, par); break;
          case 3: v_ok = attend_tile<T, D, TILE, true, 2>(sK, sK + TILE * ROWB, rows, qv, m, l, o, wb, lgs, lane, rks, rtab, low, hi, ke, vf, par); break;
          case 4: v_ok = attend_tile<T, D, TILE, true, 3>(sK, sK + TILE * ROWB, rows, qv, m, l, o, wb, lgs, lane, rks, rtab, low, hi, ke, vf, par); break;
          default: v_ok = attend_tile<T, D, TILE, true, 4>(sK, sK + TILE * ROWB, rows, qv, m, l, o, wb, lgs, lane, rks, rtab, low, hi, ke, vf, par); break;
        }
        if (!v_ok) {
          ok = false;
          if (lane == 0) atomicOr(prm.err, ERR_MBAR_TIMEOUT);
        }
        // the V half may be refilled; after a timeout it is not released
        if (lane == 0 && ok) mbar_arrive(&emptyv_bar[s]);
      } else {
        attend_tile<T, D, TILE>(sK, sK + TILE * ROWB, rows, qv, m, l, o, wb, lg + t * TILE, lane);
        // stage s may be refilled; after a timeout the stage is not released,
        // so no new copy can target memory an unfinished copy still writes
        if (lane == 0 && ok) mbar_arrive(&empty_bar[s]);
      }
    }

    merge_groups<T, D>(m, l, o);  // identical result in every row group
    // Each warp's merged (m, l, o) goes into its own first stage: every stage
    // of warp w (s % NCW == w) has been consumed, and no copy targets it, once
    // the warp has left its loop.
    auto red_of = [&](int w) { return reinterpret_cast<float*>(stage_base + static_cast<size_t>(w) * Cfg::STAGE); };
    float* myred = red_of(warp);
    if (lane == 0) {
      myred[0] = m;
      myred[1] = l;
    }
    if (grp == 0) {
#pragma unroll
      for (int e = 0; e < EPV; ++e) myred[4 + lig * EPV + e] = o[e];
    }
    cp_async_wait<0>();  // this thread's score and position copies have landed
    consumer_sync(NCW * 32);
    H2O_TL(4);
    // A pair handled by one CTA needs no cluster or distributed shared
    // memory.  In a cluster, every CTA pushes its partial softmax (m, l) into
    // each peer's xin[rank] as soon as it is merged over the warps, and the
    // other ranks then push their partial output rows into rank 0, all with
    // st.async counted on the receiver's xbar: each CTA waits only for the
    // bytes it receives, never on a cluster barrier.  Threads below D (whole
    // consumer warps) do all of a CTA's pushes.
    if (tid < D) {
      float M = kNeg;
      for (int w = 0; w < NCW; ++w) M = fmaxf(M, red_of(w)[0]);
      float Ls = 0.f;
      for (int w = 0; w < NCW; ++w) Ls = fmaf(red_of(w)[1], exp2f(red_of(w)[0] - M), Ls);
      if (S > 1) {
        cluster_wait_acquire();  // every peer has started and set up its barriers
        if (tid < S && tid != rank) {
          const uint4 v = make_uint4(__float_as_uint(M), __float_as_uint(Ls), __float_as_uint(s_self), 0u);
          st_async_v4(mapa_shared(smem_u32(&xin[rank]), tid), v, mapa_shared(smem_u32(xbar), tid));
        }
      }
      float Od = 0.f;
      for (int w = 0; w < NCW; ++w) Od = fmaf(red_of(w)[4 + tid], exp2f(red_of(w)[0] - M), Od);
      xo[tid] = Od;
      if (S > 1 && rank != 0)
        st_async_b32(mapa_shared(smem_u32(xo_in + (rank - 1) * D + tid), 0), __float_as_uint(Od),
                     mapa_shared(smem_u32(xbar), 0));
      if (tid == 0) {
        xch->m = M;
        xch->l = Ls;
        xch->s_self = s_self;
        xin[rank] = *xch;
      }
    }
  }
  const bool clustered = S > 1;
  __syncthreads();  // xo / xch / xin[rank] of this CTA are complete (all threads)
  if (clustered && !mbar_wait_cluster_bounded(xbar, 0, kWaitLimit) && tid == 0) atomicOr(prm.err, ERR_XCH_TIMEOUT);
  H2O_TL(5);

  // the pair's normaliser: merged over the cluster's CTAs, or, for a pair
  // handled by one CTA, this CTA's own (published before the barrier above)
  float M = kNeg, Ls = 0.f, sself;
  if (clustered) {
    for (int r = 0; r < S; ++r) M = fmaxf(M, xin[r].m);
    for (int r = 0; r < S; ++r) Ls = fmaf(xin[r].l, exp2f(xin[r].m - M), Ls);
    sself = xin[0].s_self;
  } else {
    M = xch->m;
    Ls = xch->l;
    sself = xch->s_self;
  }
  p = blk_int[1];
  count = blk_int[2];
  head = blk_int[3];
  const bool full = count >= C;
  const int nrows = max(min(lo + prm.chunk, count) - lo, 0);
  const float inv = 1.f / Ls;
  const float p_self = exp2f(sself - M) * inv;

  // the pair's output row (rank 0): with position rolling written once this
  // CTA's candidate is on its way to the peers (measured faster there), else
  // right away (measured faster for the plain kernel's 8-CTA clusters)
  auto write_output = [&]() {
    if (rank == 0 && tid < D) {
      float acc = xo[tid];
      if (clustered) {
        acc = 0.f;
        for (int r = 0; r < S; ++r)
          acc = fmaf(r == 0 ? xo[tid] : xo_in[(r - 1) * D + tid], exp2f(xin[r].m - M), acc);
      }
      prm.out[static_cast<size_t>(pair) * D + tid] = acc * inv;
    }
  };
  if constexpr (!ROPE) write_output();

  // probabilities -> accumulated scores, stored at once (the evicted slot's
  // score is overwritten with the newcomer's below, after the block barrier
  // that orders the two stores); local minimum candidate key
  // For a pair on one CTA, or more than two slots per thread, four slots per
  // thread and pass (the per-slot arrays start 16-byte aligned and hold a
  // multiple of four entries; the scores go out as one 16-byte store where
  // the slots' global address allows it); else one slot per thread, which
  // measured faster for the short slot ranges of 8-CTA clusters.
  const int limit = p - R;  // candidates: kept positions <= p - R outside the static pattern
  unsigned long long kmin = ~0ull;
  int smin = -1;
  if (S == 1 || nrows > 2 * NT) {
    const bool vec_store = (reinterpret_cast<uintptr_t>(prm.score + slot0) & 15u) == 0;
    for (int j0 = tid * 4; j0 < nrows; j0 += NT * 4) {
      const float4 s4 = *reinterpret_cast<const float4*>(sc + j0);
      const float4 l4 = *reinterpret_cast<const float4*>(lg + j0);
      const int4 p4 = *reinterpret_cast<const int4*>(ps + j0);
      const float sv[4] = {s4.x, s4.y, s4.z, s4.w}, lv[4] = {l4.x, l4.y, l4.z, l4.w};
      const int pv[4] = {p4.x, p4.y, p4.z, p4.w};
      float ns[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) ns[k] = sv[k] + exp2f(lv[k] - M) * inv;
      if (vec_store && j0 + 4 <= nrows) {
        *reinterpret_cast<float4*>(prm.score + slot0 + j0) = make_float4(ns[0], ns[1], ns[2], ns[3]);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (j0 + k < nrows) prm.score[slot0 + j0 + k] = ns[k];
      }
      if (full) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (j0 + k < nrows && pv[k] <= limit && !is_protected(prm.sp, pv[k])) {
            const unsigned long long key =
                (static_cast<unsigned long long>(__float_as_uint(ns[k])) << 32) | static_cast<uint32_t>(pv[k]);
            if (key < kmin) {
              kmin = key;
              smin = lo + j0 + k;
            }
          }
      }
    }
  } else {
    for (int j = tid; j < nrows; j += NT) {
      const float ns = sc[j] + exp2f(lg[j] - M) * inv;
      prm.score[slot0 + j] = ns;
      if (full && ps[j] <= limit && !is_protected(prm.sp, ps[j])) {
        const unsigned long long key =
            (static_cast<unsigned long long>(__float_as_uint(ns)) << 32) | static_cast<uint32_t>(ps[j]);
        if (key < kmin) {
          kmin = key;
          smin = lo + j;
        }
      }
    }
  }
  H2O_TL(8);
  // warp minimum, and the slot of the lane that holds it (keys are unique:
  // positions are)
  const unsigned long long wk = warp_min_key(kmin);
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
  H2O_TL(9);
  // position rolling: the candidate's rank inside the cache travels with it
  int brank = -1;
  if constexpr (ROPE) brank = bslot >= 0 ? rk[bslot - lo] : -1;

  int u, urank = brank;
  if (clustered) {
    // every thread holds this CTA's candidate (bk, bslot): thread r pushes it
    // into peer r's kin[rank]; each CTA waits for its peers' candidates
    if (tid < S && tid != rank) {
      const uint4 v = make_uint4(static_cast<uint32_t>(bk), static_cast<uint32_t>(bk >> 32),
                                 static_cast<uint32_t>(bslot), static_cast<uint32_t>(brank));
      st_async_v4(mapa_shared(smem_u32(&kin[rank]), tid), v, mapa_shared(smem_u32(kbar), tid));
    }
    H2O_TL(10);
    if constexpr (ROPE) write_output();
    if (!mbar_wait_cluster_bounded(kbar, 0, kWaitLimit) && tid == 0) atomicOr(prm.err, ERR_XCH_TIMEOUT);
    if (full) {
      unsigned long long best = ~0ull;
      u = -1;
      for (int r = 0; r < S; ++r) {
        const uint4 c = kin[r];
        const unsigned long long key = r == rank ? bk : (static_cast<unsigned long long>(c.y) << 32 | c.x);
        if (key < best) {
          best = key;
          u = r == rank ? bslot : static_cast<int>(c.z);
          urank = r == rank ? brank : static_cast<int>(c.w);
        }
      }
    } else {
      u = count;
    }
  } else {
    u = full ? bslot : count;
    if constexpr (ROPE) write_output();
  }
  if (full && u < 0 && tid == 0) atomicOr(prm.err, ERR_NO_CANDIDATE);
  H2O_TL(6);
  // Every byte pushed into this CTA has landed (both waits above) and no CTA
  // reads another's shared memory, so the CTAs of a cluster leave without a
  // cluster barrier.

  // position rolling: after an eviction the kept tokens ranked above the
  // victim move down one place and the newcomer takes the last rank, C - 1;
  // while filling, every rank stays and the newcomer takes rank `count`
  if constexpr (ROPE) {
    if (full && u >= 0) {
      const bool vec = (reinterpret_cast<uintptr_t>(prm.rank + slot0) & 15u) == 0;
      for (int j0 = tid * 4; j0 < nrows; j0 += NT * 4) {
        const int4 r4 = *reinterpret_cast<const int4*>(rk + j0);
        int rv[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (rv[k] > urank) --rv[k];
          if (lo + j0 + k == u) rv[k] = C - 1;
        }
        if (vec && j0 + 4 <= nrows) {
          *reinterpret_cast<int4*>(prm.rank + slot0 + j0) = make_int4(rv[0], rv[1], rv[2], rv[3]);
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (j0 + k < nrows) prm.rank[slot0 + j0 + k] = rv[k];
        }
      }
    }
  }
  // the new token into slot u
  if (u >= lo && u < lo + prm.chunk && u >= 0) {
    const size_t us = static_cast<size_t>(pair) * C + u;
    if (tid < 2 * LPR) {
      unsigned char* dst = static_cast<unsigned char*>(tid < LPR ? prm.K : prm.V) + us * ROWB + (tid % LPR) * 16;
      *reinterpret_cast<uint4*>(dst) = newrow;
    }
    if (tid == 0) {
      prm.pos[us] = p;
      prm.score[us] = p_self;
      if constexpr (ROPE) {
        if (!full) prm.rank[us] = count;
      }
    }
  }
  if (rank == 0 && tid == 0) {
    if (u >= 0) prm.ring[static_cast<size_t>(pair) * R + head] = u;
    *reinterpret_cast<int4*>(prm.ctr + pair) = make_int4(p + 1, full ? C : count + 1, (head + 1) % R, 0);
    if (prm.evicted) prm.evicted[pair] = full ? u : -1;
  }
  H2O_TL(7);
}

// ------------------------------------------------------------ warp per pair
// For many short pairs (thousands of (batch, head) pairs of about a hundred
// slots) a CTA per pair spends most of its short life starting up and
// finishing.  Here one warp handles a whole pair and then moves on: a grid of
// resident CTAs, grid warp w taking pairs w, w + W, w + 2W, ... (W warps in
// the grid).  Each warp feeds its own ring of stages; its lane 0 issues the
// bulk copies of the next tiles as soon as a stage is consumed, running on
// into the warp's next pair, so the copies never wait for a pair's epilogue.
// Attention, score update, argmin and overwrite of a pair are all
// warp-synchronous (shuffles, no block barrier), and a warp's ring is used by
// that warp alone, so any ring depth is safe.
constexpr int kWarpMaxStages = 8;
constexpr int kWarpMaxPairs = 64;    // pairs per warp; larger problems get a larger grid
constexpr int kWarpMaxSlots = 1024;  // slots per pair
constexpr int kWarpNW = 4;           // warps per CTA

template <typename T, int D>
struct WarpLayout {
  static constexpr int TILE = 16;
  static constexpr int STAGE = 2 * TILE * RowGeom<T, D>::ROWB;
  static constexpr size_t bars = 0;                                     // [NW][kWarpMaxStages]
  static constexpr size_t ctrs = bars + 8 * kWarpNW * kWarpMaxStages;   // [NW][kWarpMaxPairs] int4
  static constexpr size_t wbuf = ctrs + 16 * kWarpNW * kWarpMaxPairs;   // [NW][TILE] floats
  static constexpr size_t state = wbuf + 4 * kWarpNW * TILE;            // [NW][3][Cp]: logits, scores, positions
  __host__ __device__ static int cpad(int C) { return (C + 3) / 4 * 4; }
  __host__ __device__ static size_t stages(int C) {
    return (state + 12 * static_cast<size_t>(kWarpNW) * cpad(C) + 127) / 128 * 128;
  }
  __host__ __device__ static size_t bytes(int nstage, int C) {
    return stages(C) + static_cast<size_t>(kWarpNW) * nstage * STAGE;
  }
};

template <typename T, int D>
__global__ void __launch_bounds__(kWarpNW * 32, 1) decode_warp_kernel(const DecodeParams prm) {
  using Gm = RowGeom<T, D>;
  using Lay = WarpLayout<T, D>;
  constexpr int TILE = Lay::TILE, EPV = Gm::EPV, LPR = Gm::LPR, ROWB = Gm::ROWB;
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp = lane / LPR, lig = lane % LPR;
  const int C = prm.C, R = prm.R, NS = prm.nstage, pairs = prm.pairs;
  const int Cp = Lay::cpad(C);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::bars) + warp * kWarpMaxStages;
  int4* pctr = reinterpret_cast<int4*>(smem + Lay::ctrs) + warp * kWarpMaxPairs;
  float* wb = reinterpret_cast<float*>(smem + Lay::wbuf) + warp * TILE;
  float* lg = reinterpret_cast<float*>(smem + Lay::state) + static_cast<size_t>(warp) * 3 * Cp;
  float* sc = lg + Cp;
  int* ps = reinterpret_cast<int*>(sc + Cp);
  unsigned char* stg = smem + Lay::stages(C) + static_cast<size_t>(warp) * NS * Lay::STAGE;

  const int gw = blockIdx.x * kWarpNW + warp, W = gridDim.x * kWarpNW;
  const int np = gw < pairs ? (pairs - 1 - gw) / W + 1 : 0;  // pairs of this warp
  const bool ring_ok = NS >= 2 && NS <= kWarpMaxStages && np <= kWarpMaxPairs && C <= kWarpMaxSlots;
  if (np == 0) return;
  if (!ring_ok) {  // rejected on the host; a kernel given such a shape does nothing
    if (lane == 0) atomicOr(prm.err, ERR_RING_TIMEOUT);
    return;
  }
  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  const unsigned char* gK = static_cast<const unsigned char*>(prm.K);
  const unsigned char* gV = static_cast<const unsigned char*>(prm.V);
  const uint64_t policy = policy_evict_first();
  // Counters of this warp's pairs.  Cache-owned state: read before the
  // grid-dependency wait only when no earlier kernel on the stream touched
  // this cache (likewise the slot store the first copies read).
  auto load_ctrs = [&]() {
    for (int k = lane; k < np; k += 32)
      pctr[k] = *reinterpret_cast<const int4*>(prm.ctr + gw + static_cast<size_t>(k) * W);
    __syncwarp();
  };
  // Issue cursor, identical in every lane (lane 0 issues): tile t_i of the
  // warp's pair k_i; `issued` tiles so far over all the warp's pairs.  Tile
  // number n always goes to stage n % NS.
  int k_i = 0, t_i = 0, issued = 0;
  auto issue_upto = [&](int limit) {
    while (issued < limit && k_i < np) {
      const int cnt = min(max(pctr[k_i].y, 0), C);
      if (t_i * TILE >= cnt) {
        ++k_i;
        t_i = 0;
        continue;
      }
      if (lane == 0) {
        const int rows = min(TILE, cnt - t_i * TILE);
        const uint32_t bytes = static_cast<uint32_t>(rows * ROWB);
        unsigned char* st = stg + static_cast<size_t>(issued % NS) * Lay::STAGE;
        uint64_t* bar = &full[issued % NS];
        const size_t row0 = (static_cast<size_t>(gw) + static_cast<size_t>(k_i) * W) * C +
                            static_cast<size_t>(t_i) * TILE;
        mbar_arrive_expect_tx(bar, 2 * bytes);
        bulk_g2s_stream(st, gK + row0 * ROWB, bytes, bar, policy);
        bulk_g2s_stream(st + TILE * ROWB, gV + row0 * ROWB, bytes, bar, policy);
      }
      ++t_i;
      ++issued;
    }
  };
  if (lane < 3 * ((ROWB + 127) / 128)) {  // warm L2 with the first pair's q, k_new and v_new rows
    constexpr int NLINE = (ROWB + 127) / 128;
    const void* row = lane < NLINE ? prm.q : (lane < 2 * NLINE ? prm.k_new : prm.v_new);
    prefetch_l2(static_cast<const unsigned char*>(row) + static_cast<size_t>(gw) * ROWB + (lane % NLINE) * 128);
  }
  if (prm.prefetch) {
    load_ctrs();
    issue_upto(NS);
  }
  griddep_wait();  // every earlier kernel on the stream has completed
  if (!prm.prefetch) {
    load_ctrs();
    issue_upto(NS);
  }

  int consumed = 0, landed = 0;  // tiles consumed / whose copies were seen complete
  bool ok = true;
  // This lane's 16-byte slices of q, k_new and v_new, one pair ahead: the
  // next pair's are loaded while the current one streams.
  auto load_inputs = [&](int pr, uint4& q4, uint4& k4, uint4& v4) {
    const size_t off = static_cast<size_t>(pr) * ROWB + lig * 16;
    q4 = *reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(prm.q) + off);
    k4 = *reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(prm.k_new) + off);
    v4 = *reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(prm.v_new) + off);
  };
  uint4 q4, k4, v4, nq4, nk4, nv4;
  load_inputs(gw, q4, k4, v4);
  for (int k = 0; k < np; ++k) {
    const int pr = gw + k * W;
    const int4 c4 = pctr[k];
    const int p = c4.x, count = min(max(c4.y, 0), C), head = c4.z;
    const size_t slot0 = static_cast<size_t>(pr) * C;
    // this pair's scores and positions, needed from the epilogue on
    for (int j = lane; j < count; j += 32) {
      cp_async4(sc + j, prm.score + slot0 + j);
      cp_async4(ps + j, prm.pos + slot0 + j);
    }
    cp_async_commit();
    if (k + 1 < np) load_inputs(pr + W, nq4, nk4, nv4);
    // q (pre-scaled into the base-2 domain); the new token attends to
    // itself: row group 0 starts from it
    float qv[EPV], kf[EPV], o[EPV];
    Vec16<T>::unpack(q4, qv);
#pragma unroll
    for (int e = 0; e < EPV; ++e) qv[e] *= prm.qscale;
    Vec16<T>::unpack(k4, kf);
    float a = 0.f;
#pragma unroll
    for (int e = 0; e < EPV; ++e) a = fmaf(qv[e], kf[e], a);
#pragma unroll
    for (int off = LPR / 2; off >= 1; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
    const float s_self = a;
    float m = kNeg, l = 0.f;
#pragma unroll
    for (int e = 0; e < EPV; ++e) o[e] = 0.f;
    if (grp == 0) {
      Vec16<T>::unpack(v4, o);
      m = s_self;
      l = 1.f;
    }
    if (k == 0) griddep_launch();  // this step's first inputs are loaded

    const int nt = (count + TILE - 1) / TILE;
    for (int t = 0; t < nt; ++t) {
      const int s = consumed % NS;
      if (ok) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait_bounded(&full[s], static_cast<uint32_t>((consumed / NS) & 1), kWaitLimit));
        if (ok)
          ++landed;
        else if (lane == 0)
          atomicOr(prm.err, ERR_MBAR_TIMEOUT);
      }
      const unsigned char* sK = stg + static_cast<size_t>(s) * Lay::STAGE;
      const int rows = ok ? min(TILE, count - t * TILE) : 0;
      attend_tile<T, D, TILE>(sK, sK + TILE * ROWB, rows, qv, m, l, o, wb, lg + t * TILE, lane);
      ++consumed;
      if (ok) issue_upto(consumed + NS);  // the stage just read may be refilled
    }

    merge_groups<T, D>(m, l, o);
    const float inv = 1.f / l;
    const float p_self = exp2f(s_self - m) * inv;
    if (ok && grp == 0) {
      float* dst = prm.out + static_cast<size_t>(pr) * D + lig * EPV;
#pragma unroll
      for (int e = 0; e < EPV; e += 4)
        *reinterpret_cast<float4*>(dst + e) = make_float4(o[e] * inv, o[e + 1] * inv, o[e + 2] * inv, o[e + 3] * inv);
    }
    // probabilities -> accumulated scores, stored at once (after a failed
    // wait nothing is stored; the evicted slot's score is overwritten with
    // the newcomer's below, in program order after a warp barrier); the
    // lowest candidate key (score bits, position) among kept positions <= p - R
    cp_async_wait<0>();
    __syncwarp();
    const bool fullc = count >= C;
    const int limit = p - R;
    unsigned long long kmin = ~0ull;
    int smin = -1;
    for (int j = lane; j < count; j += 32) {
      const float ns = sc[j] + exp2f(lg[j] - m) * inv;
      if (ok) prm.score[slot0 + j] = ns;
      if (fullc && ps[j] <= limit && !is_protected(prm.sp, ps[j])) {
        const unsigned long long key =
            (static_cast<unsigned long long>(__float_as_uint(ns)) << 32) | static_cast<uint32_t>(ps[j]);
        if (key < kmin) {
          kmin = key;
          smin = j;
        }
      }
    }
    const unsigned long long wk = warp_min_key(kmin);
    const unsigned holder = __ballot_sync(0xffffffffu, kmin == wk && kmin != ~0ull);
    const int wslot = __shfl_sync(0xffffffffu, smin, holder ? __ffs(holder) - 1 : 0);
    const int u = fullc ? (holder ? wslot : -1) : count;
    __syncwarp();
    if (ok) {
      if (fullc && u < 0 && lane == 0) atomicOr(prm.err, ERR_NO_CANDIDATE);
      if (u >= 0) {
        // the new row from the slices already in registers: row group 0
        // writes K, group 1 writes V (one group covering the row: both)
        const size_t us = (slot0 + u) * ROWB + lig * 16;
        if (grp == 0) *reinterpret_cast<uint4*>(static_cast<unsigned char*>(prm.K) + us) = k4;
        if (grp == (LPR == 32 ? 0 : 1)) *reinterpret_cast<uint4*>(static_cast<unsigned char*>(prm.V) + us) = v4;
        if (lane == 0) {
          prm.pos[slot0 + u] = p;
          prm.score[slot0 + u] = p_self;
        }
      }
      if (lane == 0) {
        if (u >= 0) prm.ring[static_cast<size_t>(pr) * R + head] = u;
        *reinterpret_cast<int4*>(prm.ctr + pr) = make_int4(p + 1, fullc ? C : count + 1, (head + 1) % R, 0);
        if (prm.evicted) prm.evicted[pr] = fullc ? u : -1;
      }
    }
    __syncwarp();  // sc, ps and lg are refilled for the next pair
    q4 = nq4;
    k4 = nk4;
    v4 = nv4;
  }
  // no copy may still be landing in shared memory when the warp exits
  if (lane == 0)
    for (int n = landed; n < issued; ++n)
      if (!mbar_wait_bounded(&full[n % NS], static_cast<uint32_t>((n / NS) & 1), kWaitLimit))
        atomicOr(prm.err, ERR_RING_TIMEOUT);
}

template <typename T, int D>
struct WarpKern {
  using Lay = WarpLayout<T, D>;
  static constexpr auto fn = decode_warp_kernel<T, D>;

  static cudaError_t attrs() {
    size_t most = Lay::bytes(kWarpMaxStages, kWarpMaxSlots);
    if (most > 227 * 1024) most = 227 * 1024;
    return kernel_attrs(reinterpret_cast<const void*>(fn), most, false);
  }
  // CTAs resident per SM (0 = cannot launch)
  static int per_sm(int nstage, int C) {
    const size_t bytes = Lay::bytes(nstage, C);
    if (bytes > 227 * 1024 || attrs() != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kWarpNW * 32, bytes) != cudaSuccess) return 0;
    return n;
  }
  static cudaError_t launch(const DecodeParams& prm, int ctas, cudaStream_t s) {
    cudaError_t e = attrs();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas, 1, 1);
    cfg.blockDim = dim3(kWarpNW * 32, 1, 1);
    cfg.dynamicSmemBytes = Lay::bytes(prm.nstage, prm.C);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, prm);
  }
};

template <typename T, int D, int NCW, bool ROPE>
struct Kern {
  static constexpr int TILE = 16;
  using Cfg = DecodeCfg<T, D, NCW, TILE, producer_warps(ROPE)>;
  using Lay = Layout<D, NCW, TILE, Cfg::STAGE, ROPE>;
  static constexpr auto fn = decode_kernel<T, D, NCW, TILE, ROPE>;

  // entries: position rolling's rotation-table entries (0 when off)
  static size_t smem(int nstage, int chunk, int splits, int entries) {
    return Lay::bytes(nstage, chunk, splits, entries);
  }

  static cudaError_t attrs() {
    // raised once for the largest configuration, so later launches (also
    // inside stream capture) make no attribute calls
    size_t most = Lay::bytes(kMaxStages, kMaxChunk, 16, rope_entries_for(65536, kRopeMinBits, kRopeMinBits));
    if (most > 227 * 1024) most = 227 * 1024;
    return kernel_attrs(reinterpret_cast<const void*>(fn), most, true);
  }

  static cudaError_t launch(const DecodeParams& prm, int pairs, int splits, cudaStream_t s) {
    cudaError_t e = attrs();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(splits, pairs, 1);
    cfg.blockDim = dim3(Cfg::NT, 1, 1);
    cfg.dynamicSmemBytes =
        smem(prm.nstage, prm.chunk, splits,
             prm.rope ? rope_entries_for(prm.C, prm.rope_low_bits, prm.rope_hi_bits) : 0);
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
  static int resident(int splits, int nstage, int chunk, int pairs, int sms, int entries) {
    if (attrs() != cudaSuccess) return 0;
    const size_t bytes = smem(nstage, chunk, splits, entries);
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

template <int NCW, bool ROPE, typename F>
auto dispatch_ncw(int dtype, int D, F&& f) -> decltype(f(Kern<__half, 128, NCW, ROPE>{})) {
  if (dtype == 0 && D == 128) return f(Kern<__half, 128, NCW, ROPE>{});
  if (dtype == 0 && D == 64) return f(Kern<__half, 64, NCW, ROPE>{});
  if (dtype == 1 && D == 128) return f(Kern<float, 128, NCW, ROPE>{});
  return f(Kern<float, 64, NCW, ROPE>{});
}
// the kernel instance for a dtype, head width, cluster size and position rolling
template <typename F>
auto dispatch(int dtype, int D, int splits, bool rope, F&& f) -> decltype(f(Kern<__half, 128, 4, false>{})) {
  if (rope)
    return splits > 1 ? dispatch_ncw<consumer_warps(2, true), true>(dtype, D, f)
                      : dispatch_ncw<consumer_warps(1, true), true>(dtype, D, f);
  return splits > 1 ? dispatch_ncw<consumer_warps(2), false>(dtype, D, f)
                    : dispatch_ncw<consumer_warps(1), false>(dtype, D, f);
}

}  // namespace

int decode_max_chunk() { return kMaxChunk; }

int decode_chunk(int C, int splits) { return chunk_for(C, splits); }

int decode_max_stages() { return kMaxStages; }
int decode_stage_multiple(int splits, bool rope) { return consumer_warps(splits, rope); }

int device_sms() {
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return sms;
}

int decode_resident(int dtype, int D, int splits, int nstage, int chunk, int pairs, int rope_entries) {
  const int sms = device_sms();
  const int r = dispatch(dtype, D, splits, rope_entries > 0, [&](auto k) {
    return decltype(k)::resident(splits, nstage, chunk, pairs, sms, rope_entries);
  });
  cudaGetLastError();
  return r;
}

// Default launch shape.  Consecutive decode steps of different layers
// overlap: the next kernel's CTAs start filling their rings while this one
// finishes, so one step should take about 1.7 CTAs per SM (the largest
// cluster size whose grid stays within that, each CTA keeping at least 32
// slots), with a 12-stage ring (two or three stages in flight per consumer warp)
// when two such CTAs fit on an SM.  Grids that need several waves anyway
// (many pairs) use rings of one stage per consumer warp so that more CTAs
// are resident.
// Many short pairs (at least four per SM, each within the warp kernel's slot
// limit) go to the warp-per-pair kernel.  More resident warps beat deeper
// rings, so its ring is the deepest that still leaves as many resident warps
// as there are pairs, up to the count the shallowest ring allows.
int decode_warp_default_stages(int dtype, int D, int C, int pairs) {
  const long long most = static_cast<long long>(decode_warp_resident(dtype, D, 2, C)) * kWarpNW;
  const long long want = pairs < most ? pairs : most;
  for (int st = kWarpMaxStages; st > 2; --st)
    if (static_cast<long long>(decode_warp_resident(dtype, D, st, C)) * kWarpNW >= want) return st;
  return 2;
}

DecodeShape decode_pick_shape(int dtype, int D, int pairs, int C, int rope_entries) {
  const bool rope = rope_entries > 0;
  const int sms = device_sms();
  // position rolling runs on the cluster kernel only
  if (!rope && sms > 0 && C <= kWarpMaxSlots && pairs >= 4 * sms && decode_warp_resident(dtype, D, 2, C) > 0) {
    DecodeShape w;
    w.splits = kDecodeWarpPerPair;
    w.stages = decode_warp_default_stages(dtype, D, C, pairs);
    return w;
  }
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
  const int ncw = consumer_warps(sh.splits, rope);
  sh.stages = ncw;
  if (ctas <= 2LL * sms) {
    const int ch = chunk_for(C, sh.splits);
    const int deep = ncw <= 12 ? 12 / ncw * ncw : ncw;
    for (int st : {deep, ncw == 4 ? 8 : ncw}) {
      const int res = decode_resident(dtype, D, sh.splits, st, ch, pairs, rope_entries);
      if (res >= 2 * sms || static_cast<long long>(res) >= ctas) {
        sh.stages = st;
        break;
      }
    }
  }
  return sh;
}

RopeRadix decode_pick_rope_radix(int dtype, int D, int pairs, int C) {
  // candidates by levels, then entries; the smallest tables set the bar
  struct Cand {
    int levels, entries, low, hi;
  };
  Cand best{0, 0, 0, 0}, least{0, 0, 0, 0};
  std::vector<Cand> all;
  for (int low = kRopeMinBits; low <= kRopeMaxBits; ++low)
    for (int hi = kRopeMinBits; hi <= kRopeMaxBits; ++hi)
      all.push_back({rope_levels_for(C, low, hi), rope_entries_for(C, low, hi), low, hi});
  std::sort(all.begin(), all.end(), [](const Cand& a, const Cand& b) {
    if (a.levels != b.levels) return a.levels < b.levels;
    if (a.entries != b.entries) return a.entries < b.entries;
    return a.low != b.low ? a.low < b.low : a.hi < b.hi;
  });
  for (const Cand& c : all)
    if (least.entries == 0 || c.entries < least.entries) least = c;
  auto resident = [&](int entries) {
    const DecodeShape sh = decode_pick_shape(dtype, D, pairs, C, entries);
    return std::make_pair(sh.stages, decode_resident(dtype, D, sh.splits, sh.stages, chunk_for(C, sh.splits), pairs,
                                                     entries));
  };
  const auto bar = resident(least.entries);
  best = least;
  for (const Cand& c : all) {
    const auto r = resident(c.entries);
    if (r.first >= bar.first && r.second >= bar.second) {
      best = c;
      break;
    }
  }
  return RopeRadix{best.low, best.hi};
}

int decode_warp_max_slots() { return kWarpMaxSlots; }
int decode_warp_min_stages() { return 2; }
int decode_warp_max_stages() { return kWarpMaxStages; }

int decode_warp_resident(int dtype, int D, int nstage, int C) {
  if (nstage < 2 || nstage > kWarpMaxStages || C > kWarpMaxSlots) return 0;
  const int sms = device_sms();
  int per = 0;
  if (dtype == 0 && D == 128) per = WarpKern<__half, 128>::per_sm(nstage, C);
  else if (dtype == 0 && D == 64) per = WarpKern<__half, 64>::per_sm(nstage, C);
  else if (dtype == 1 && D == 128) per = WarpKern<float, 128>::per_sm(nstage, C);
  else per = WarpKern<float, 64>::per_sm(nstage, C);
  cudaGetLastError();
  return per * sms;
}

namespace {
// resident CTAs of the warp-per-pair kernel for a shape, looked up once
int warp_grid(int dtype, int D, int nstage, int C, int pairs) {
  static std::mutex mu;
  static std::map<std::array<int, 5>, int> known;
  int dev = 0;
  cudaGetDevice(&dev);
  const std::array<int, 5> key{dtype, D, nstage, C, dev};
  int res;
  {
    std::lock_guard<std::mutex> g(mu);
    auto it = known.find(key);
    if (it != known.end()) {
      res = it->second;
    } else {
      res = decode_warp_resident(dtype, D, nstage, C);
      known[key] = res;
    }
  }
  const int need = (pairs + kWarpNW - 1) / kWarpNW;                           // one pair per warp
  const int least = (pairs + kWarpNW * kWarpMaxPairs - 1) / (kWarpNW * kWarpMaxPairs);  // pair-list bound
  const int g = res < need ? res : need;
  return g > least ? g : least;
}
}  // namespace

cudaError_t launch_decode(const DecodeParams& prm, int dtype, int D, int pairs, int splits, cudaStream_t s) {
  if ((dtype != 0 && dtype != 1) || (D != 64 && D != 128)) return cudaErrorInvalidValue;
  if (splits == kDecodeWarpPerPair) {
    if (prm.rope != nullptr) return cudaErrorInvalidValue;  // position rolling: cluster kernel only
    if (prm.C > kWarpMaxSlots || prm.nstage < 2 || prm.nstage > kWarpMaxStages) return cudaErrorInvalidValue;
    const int ctas = warp_grid(dtype, D, prm.nstage, prm.C, pairs);
    if (ctas <= 0) return cudaErrorInvalidConfiguration;
    if (dtype == 0 && D == 128) return WarpKern<__half, 128>::launch(prm, ctas, s);
    if (dtype == 0 && D == 64) return WarpKern<__half, 64>::launch(prm, ctas, s);
    if (dtype == 1 && D == 128) return WarpKern<float, 128>::launch(prm, ctas, s);
    return WarpKern<float, 64>::launch(prm, ctas, s);
  }
  if (prm.rope != nullptr &&
      (prm.rank == nullptr || prm.rope_low_bits < kRopeMinBits || prm.rope_low_bits > kRopeMaxBits ||
       prm.rope_hi_bits < kRopeMinBits || prm.rope_hi_bits > kRopeMaxBits ||
       prm.rope_levels != rope_levels_for(prm.C, prm.rope_low_bits, prm.rope_hi_bits) || prm.rope_levels > 5))
    return cudaErrorInvalidValue;
  return dispatch(dtype, D, splits, prm.rope != nullptr,
                  [&](auto k) { return decltype(k)::launch(prm, pairs, splits, s); });
}

int decode_threads(int splits, bool rope) { return (consumer_warps(splits, rope) + producer_warps(rope)) * 32; }

#ifdef H2O_DECODE_TIMELINE
cudaError_t decode_timeline_read(void* dst, size_t bytes) {
  const size_t n = bytes < sizeof(g_decode_tl) ? bytes : sizeof(g_decode_tl);
  return cudaMemcpyFromSymbol(dst, g_decode_tl, n);
}
#endif

}  // namespace h2o
