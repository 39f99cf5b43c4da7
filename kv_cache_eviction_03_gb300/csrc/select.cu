// H2O prefill, part 2: keep rule and slot layout.
//
// Method: "H2O: Heavy-Hitter Oracle ... 深度解读报告", section 3.4: a prompt
// longer than the cache keeps `heavy` heavy hitters plus the `recent` most
// recent tokens, a shorter one keeps everything; the cache is preallocated
// and laid out as a heavy-hitter region followed by the recent region, the
// latter used as a circular queue.
//
// Heavy hitters are the `heavy` largest keys (colsum_j, j) among positions
// j < L - recent (larger position kept on equal scores, i.e. the same total
// order under which decode evicts the minimum).  Positions of a static
// pattern (section 4.5, Table 2; at most `heavy` of them) rank above every
// score, so they are kept first and the heavy hitters fill the rest.  One CTA per pair finds the
// threshold with an MSB-first radix select on the float bits (non-negative
// floats order like their bit patterns), then compacts the kept positions in
// ascending order with block-wide ballot scans and gathers their K/V rows
// into slots 0..heavy-1 with 16-byte vector copies; the recent window goes to
// slots heavy..C-1.
#include <cuda_fp16.h>

#include "h2o_internal.cuh"
#include "ptx.cuh"

namespace h2o {
namespace {

constexpr int NT = 512;
constexpr int NW = NT / 32;

struct Scan {
  unsigned warp_tot[NW];
  unsigned total;
};

// exclusive prefix count of `flag` over the block, in thread order; returns
// the prefix and sets *total (block-wide count).  Contains __syncthreads.
__device__ __forceinline__ unsigned block_scan(bool flag, Scan& sh, unsigned* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned b = __ballot_sync(0xffffffffu, flag);
  const unsigned in_warp = __popc(b & ((1u << lane) - 1u));
  if (lane == 0) sh.warp_tot[warp] = __popc(b);
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned run = 0;
    for (int w = 0; w < NW; ++w) {
      const unsigned t = sh.warp_tot[w];
      sh.warp_tot[w] = run;
      run += t;
    }
    sh.total = run;
  }
  __syncthreads();
  const unsigned r = sh.warp_tot[warp] + in_warp;
  *total = sh.total;
  __syncthreads();
  return r;
}

// copy `n` rows listed in (src_pos, dst_slot) from the prompt into the slot
// store; each thread loads its 16-byte pieces of four rows before storing
// them, so four rows' loads are in flight at once
template <int ROWB>
__device__ __forceinline__ void copy_rows(const unsigned char* srcK, const unsigned char* srcV, unsigned char* dstK,
                                          unsigned char* dstV, const int* src_pos, const int* dst_slot, int n) {
  constexpr int LPR = ROWB / 16;
  constexpr int RPI = 32 / LPR;
  constexpr int STEP = NW * RPI, UNROLL = 4;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp = lane / LPR, lig = lane % LPR;
  for (int i0 = warp * RPI + grp; i0 < n; i0 += UNROLL * STEP) {
    uint4 kv[UNROLL], vv[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int i = i0 + u * STEP;
      if (i < n) {
        const size_t so = static_cast<size_t>(src_pos[i]) * ROWB + lig * 16;
        kv[u] = *reinterpret_cast<const uint4*>(srcK + so);
        vv[u] = *reinterpret_cast<const uint4*>(srcV + so);
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int i = i0 + u * STEP;
      if (i < n) {
        const size_t dofs = static_cast<size_t>(dst_slot[i]) * ROWB + lig * 16;
        *reinterpret_cast<uint4*>(dstK + dofs) = kv[u];
        *reinterpret_cast<uint4*>(dstV + dofs) = vv[u];
      }
    }
  }
}

// The digit d of this radix pass: the largest d >= 1 whose bins d..255 hold
// at least k keys (d = 0 if none does), with cum = the keys in bins above d.
// Warp 0 does it: lane l sums bins 255-8l .. 248-8l, a shuffle scan finds
// the lane where the running count reaches k, and that lane walks its bins
// and publishes prefix | d << shift, k - cum and the count in bin d.
__device__ __forceinline__ void pick_digit(const unsigned* hist, unsigned k, unsigned prefix, int shift,
                                           unsigned* s_prefix, unsigned* s_k, unsigned* s_eq) {
  const int lane = threadIdx.x & 31;
  const int top = 255 - 8 * lane;
  unsigned loc = 0;
#pragma unroll
  for (int x = 0; x < 8; ++x) loc += hist[top - x];
  unsigned inc = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  const unsigned exc = inc - loc;
  const unsigned who = __ballot_sync(0xffffffffu, exc < k && inc >= k);
  const int owner = who ? __ffs(who) - 1 : 31;
  if (lane == owner) {
    unsigned cum = exc, d = 0;
    for (int x = 0; x < 8; ++x) {
      const int dd = top - x;
      if (dd == 0) break;
      if (cum + hist[dd] >= k) {
        d = static_cast<unsigned>(dd);
        break;
      }
      cum += hist[dd];
    }
    *s_prefix = prefix | (d << shift);
    *s_k = k - cum;
    *s_eq = hist[d];
  }
}

// Selection key of position j: the bits of its (non-negative) column sum, or
// those of +infinity for a protected position, above every finite score.
__device__ __forceinline__ unsigned key_bits(const float* colsum, const StaticPattern& sp, int j) {
  return is_protected(sp, j) ? 0x7F800000u : __float_as_uint(colsum[j]);
}

template <int ROWB>
__global__ void __launch_bounds__(NT, 2) select_kernel(const SelectParams prm) {
  __shared__ unsigned hist[256];
  __shared__ Scan scan;
  __shared__ int list_pos[NT];
  __shared__ int list_slot[NT];
  __shared__ unsigned s_prefix, s_k, s_eq;
  const int tid = threadIdx.x;
  const int pair = blockIdx.x;
  const int LS = prm.L, heavy = prm.heavy, R = prm.recent, C = prm.C;  // LS: row stride
  const float* colsum = prm.colsum + static_cast<size_t>(pair) * LS;
  const unsigned char* srcK = static_cast<const unsigned char*>(prm.k) + static_cast<size_t>(pair) * LS * ROWB;
  const unsigned char* srcV = static_cast<const unsigned char*>(prm.v) + static_cast<size_t>(pair) * LS * ROWB;
  unsigned char* dstK = static_cast<unsigned char*>(prm.K) + static_cast<size_t>(pair) * C * ROWB;
  unsigned char* dstV = static_cast<unsigned char*>(prm.V) + static_cast<size_t>(pair) * C * ROWB;
  float* score = prm.score + static_cast<size_t>(pair) * C;
  int* pos = prm.pos + static_cast<size_t>(pair) * C;

  griddep_wait();
  const int L = pair_len(prm.lens, prm.heads, LS, pair);  // this pair's prompt length

  int n_keep;
  if (L <= C) {
    // keep everything: slot j <- position j
    n_keep = L;
    for (int j0 = 0; j0 < L; j0 += NT) {
      const int j = j0 + tid;
      if (j < L) {
        list_pos[tid] = j;
        list_slot[tid] = j;
        score[j] = colsum[j];
        pos[j] = j;
      }
      __syncthreads();
      copy_rows<ROWB>(srcK, srcV, dstK, dstV, list_pos, list_slot, min(NT, L - j0));
      __syncthreads();
    }
  } else {
    const int n = L - R;  // candidates: positions 0..n-1 (n > heavy)
    n_keep = C;
    if (heavy > 0) {
      // radix select: threshold bits T of the heavy-th largest score
      unsigned prefix = 0, mask = 0, k = static_cast<unsigned>(heavy), eq = 0;
      for (int shift = 24; shift >= 0; shift -= 8) {
        for (int b = tid; b < 256; b += NT) hist[b] = 0;
        __syncthreads();
        for (int j = tid; j < n; j += NT) {
          const unsigned bits = key_bits(colsum, prm.sp, j);
          if ((bits & mask) == prefix) atomicAdd(&hist[(bits >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (tid < 32) pick_digit(hist, k, prefix, shift, &s_prefix, &s_k, &s_eq);
        __syncthreads();
        prefix = s_prefix;
        k = s_k;
        eq = s_eq;
        mask |= 255u << shift;
        __syncthreads();
      }
      // keep: bits > T, or bits == T and among the k highest positions of those
      unsigned base_eq = 0, base_keep = 0;
      for (int j0 = 0; j0 < n; j0 += NT) {
        const int j = j0 + tid;
        const unsigned bits = j < n ? key_bits(colsum, prm.sp, j) : 0u;
        const bool is_eq = j < n && bits == prefix;
        unsigned tot_eq, tot_keep;
        const unsigned eq_rank = base_eq + block_scan(is_eq, scan, &tot_eq);
        const bool keep = j < n && (bits > prefix || (is_eq && eq_rank >= eq - k));
        const unsigned idx = block_scan(keep, scan, &tot_keep);
        if (base_keep + tot_keep > static_cast<unsigned>(heavy)) {
          // more keys than heavy slots: the threshold search failed; flag it
          // and keep the slot writes inside this pair's heavy region
          if (tid == 0) atomicOr(prm.err, ERR_SELECT);
          tot_keep = base_keep < static_cast<unsigned>(heavy) ? heavy - base_keep : 0u;
        }
        if (keep && idx < tot_keep) {
          const int slot = static_cast<int>(base_keep + idx);
          list_pos[idx] = j;
          list_slot[idx] = slot;
          score[slot] = colsum[j];
          pos[slot] = j;
        }
        __syncthreads();
        copy_rows<ROWB>(srcK, srcV, dstK, dstV, list_pos, list_slot, static_cast<int>(tot_keep));
        __syncthreads();
        base_eq += tot_eq;
        base_keep += tot_keep;
      }
      if (tid == 0 && base_keep != static_cast<unsigned>(heavy)) atomicOr(prm.err, ERR_SELECT);
    }
    // recent window: slot heavy + r <- position n + r
    for (int r0 = 0; r0 < R; r0 += NT) {
      const int r = r0 + tid;
      if (r < R) {
        list_pos[tid] = n + r;
        list_slot[tid] = heavy + r;
        score[heavy + r] = colsum[n + r];
        pos[heavy + r] = n + r;
      }
      __syncthreads();
      copy_rows<ROWB>(srcK, srcV, dstK, dstV, list_pos, list_slot, min(NT, R - r0));
      __syncthreads();
    }
  }
  for (int s = n_keep + tid; s < C; s += NT) {
    score[s] = 0.f;
    pos[s] = -1;
  }
  // recent ring (oldest first) and counters
  int* ring = prm.ring + static_cast<size_t>(pair) * R;
  int head;
  if (L > C) {
    for (int r = tid; r < R; r += NT) ring[r] = heavy + r;
    head = 0;
  } else if (L >= R) {
    for (int r = tid; r < R; r += NT) ring[r] = L - R + r;
    head = 0;
  } else {
    for (int r = tid; r < R; r += NT) ring[r] = r < L ? r : -1;
    head = L;
  }
  if (tid == 0) {
    PairCtr c;
    c.p = L;
    c.count = n_keep;
    c.head = head;
    c.pad = 0;
    prm.ctr[pair] = c;
  }
  griddep_launch();
}

__global__ void reset_kernel(PairCtr* ctr, int* pos, float* score, int* ring, int pairs, int C, int R) {
  griddep_wait();
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  const size_t t0 = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
  const size_t nc = static_cast<size_t>(pairs) * C;
  for (size_t i = t0; i < nc; i += stride) {
    pos[i] = -1;
    score[i] = 0.f;
  }
  const size_t nr = static_cast<size_t>(pairs) * R;
  for (size_t i = t0; i < nr; i += stride) ring[i] = -1;
  for (size_t i = t0; i < static_cast<size_t>(pairs); i += stride) {
    PairCtr c;
    c.p = 0;
    c.count = 0;
    c.head = 0;
    c.pad = 0;
    ctr[i] = c;
  }
}

template <typename Kern, typename P>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, cudaStream_t s, const P& prm) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, prm);
}

}  // namespace

cudaError_t launch_prefill_select(const SelectParams& prm, int dtype, int D, int pairs, cudaStream_t s) {
  const int rowb = D * (dtype == 0 ? 2 : 4);
  const dim3 grid(pairs), block(NT);
  switch (rowb) {
    case 128: return launch_pdl(select_kernel<128>, grid, block, s, prm);
    case 256: return launch_pdl(select_kernel<256>, grid, block, s, prm);
    case 512: return launch_pdl(select_kernel<512>, grid, block, s, prm);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_reset(PairCtr* ctr, int* pos, float* score, int* ring, int pairs, int C, int R,
                         cudaStream_t s) {
  const size_t work = static_cast<size_t>(pairs) * (C > R ? C : R);
  const int blocks = static_cast<int>(work < 256 * 2048 ? (work + 255) / 256 : 2048);
  reset_kernel<<<blocks, 256, 0, s>>>(ctr, pos, score, ring, pairs, C, R);
  return cudaGetLastError();
}

}  // namespace h2o
