// The split-KV tile schedule as a device function of one CTA, shared by the
// stand-alone schedule kernel and by the extra CTA that computes it inside an
// absorption's launch.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mla_kernels.h"

namespace mla {

// get_mla_metadata's role ("MLA 推理：两条计算路径与 FlashMLA", FlashMLA paragraph):
// from the sequence lengths alone, decide which KV pages each part (cluster)
// processes; at most `hbm_parts` parts are used, since that many already keep HBM
// busy, unless using all parts is estimated to be faster even with the splits it
// causes (`split_cost` pages per extra segment).  One CTA.  Every request is laid out
// on a line of cost positions: F set-up positions, then one position per page; request b
// occupies [C[b], C[b+1]).  The
// line is cut into P_eff equal pieces of T = ceil(C[B] / P_eff) positions, part p
// taking the pages whose positions lie in [p T, (p + 1) T).  The costs are
// prefix-summed by all threads; each part then finds its first and last page with
// two binary searches, independently of the other parts.
// Exclusive prefix sum of one value per thread over the block (kT threads): warp
// shuffles, then one warp over the warp totals.  `scratch` holds kT / 32 + 1 entries;
// the block total is returned in *total.
template <int kT>
__device__ __forceinline__ int64_t block_exclusive_scan(int64_t v, int64_t* scratch, int64_t* total) {
  static_assert(kT % 32 == 0 && kT / 32 <= 32, "scan shape");
  constexpr int kWarps = kT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t x = v;   // inclusive scan within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();   // scratch may still be read by a previous scan
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int64_t w = lane < kWarps ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kWarps) scratch[lane] = w;          // inclusive warp prefix
    if (lane == kWarps - 1) scratch[kWarps] = w;   // block total
  }
  __syncthreads();
  const int64_t before = warp > 0 ? scratch[warp - 1] : 0;
  *total = scratch[kWarps];
  return before + x - v;
}

// The whole block (kT threads) computes the schedule; sched_c holds B + 1 int64 and
// sched_nb B int32 of shared memory, s_scan kT / 32 + 1 int64.
template <int kT>
__device__ void schedule_body(const int32_t* seqlens, int B, int num_parts, int fixed_cost, int hbm_parts,
                              int split_cost, int32_t* meta, int32_t* num_splits, int64_t* sched_c, int32_t* sched_nb,
                              int64_t* s_scan) {
  const int tid = threadIdx.x;
  const int64_t F = fixed_cost;
  const int chunk = (B + kT - 1) / kT;
  const int lo = min(B, tid * chunk), hi = min(B, lo + chunk);
  // 1. page counts, per-thread sums of the costs, block-wide exclusive scan, C
  int64_t sum = 0;
  for (int i = lo; i < hi; ++i) {
    const int L = seqlens[i];
    const int nb = L > 0 ? (L + kPageTokens - 1) / kPageTokens : 0;
    sched_nb[i] = nb;
    sum += nb > 0 ? nb + F : 0;
  }
  int64_t block_total;
  int64_t run = block_exclusive_scan<kT>(sum, s_scan, &block_total);
  if (tid == 0) sched_c[0] = 0;
  for (int i = lo; i < hi; ++i) {
    run += sched_nb[i] > 0 ? sched_nb[i] + F : 0;
    sched_c[i + 1] = run;
  }
  __syncthreads();
  const int64_t total = sched_c[B];
  int p_eff = max(1, min(num_parts, hbm_parts));
  // segments of request i when parts hold T positions each
  auto segments = [&](int i, int64_t T) -> int64_t {
    const int nb = sched_nb[i];
    return nb > 0 ? (sched_c[i] + F + nb - 1) / T - (sched_c[i] + F) / T + 1 : 0;
  };
  if (split_cost > 0 && total > 0 && num_parts > p_eff) {
    int64_t best_est = -1;
    int best_p = p_eff;
    const int cand[2] = {p_eff, num_parts};
    for (int c = 0; c < 2; ++c) {
      const int pe = cand[c];
      const int64_t Tc = (total + pe - 1) / pe;
      int64_t extra = 0;
      for (int i = lo; i < hi; ++i) extra += sched_nb[i] > 0 ? segments(i, Tc) - 1 : 0;
      int64_t all_extra;
      block_exclusive_scan<kT>(extra, s_scan, &all_extra);
      const int64_t est = Tc + static_cast<int64_t>(split_cost) * ((all_extra + pe - 1) / pe);
      if (best_est < 0 || est < best_est) best_est = est, best_p = pe;
    }
    p_eff = best_p;
  }
  const int64_t T = (total + p_eff - 1) / p_eff;
  // first index b in [0, B) with C[b + 1] > x (C[1..B] is non-decreasing); B if none
  auto first_above = [&](int64_t x) {
    int l = 0, h = B;
    while (l < h) {
      const int m = (l + h) >> 1;
      if (sched_c[m + 1] > x) h = m; else l = m + 1;
    }
    return l;
  };
  // 2. one metadata record per part
  for (int p = tid; p < num_parts; p += kT) {
    int32_t m[kMetaInts] = {-1, 0, 0, 0, 0, 0, 0, 0};
    const int64_t plo = static_cast<int64_t>(p) * T, phi = plo + T;
    if (total > 0 && p < p_eff && plo < total) {
      const int bf = first_above(plo);
      const int64_t kf0 = plo - sched_c[bf] - F;
      const int64_t kf = kf0 > 0 ? kf0 : 0;
      if (sched_c[bf] + F + kf < phi) {
        // the last non-empty request whose first page lies before phi: x = the number of
        // requests b with C[b] + F < phi; the last page before C[x] belongs to it
        int l = 0, h = B;
        while (l < h) {
          const int mid = (l + h) >> 1;
          if (sched_c[mid] + F >= phi) h = mid; else l = mid + 1;
        }
        const int bl = first_above(sched_c[l] - 1);
        const int64_t ke0 = phi - sched_c[bl] - F;
        const int64_t ke = ke0 < sched_nb[bl] ? ke0 : static_cast<int64_t>(sched_nb[bl]);
        m[0] = bf;
        m[1] = static_cast<int32_t>(kf);
        m[2] = bl;
        m[3] = static_cast<int32_t>(ke);
        m[4] = static_cast<int32_t>(p - (sched_c[bf] + F) / T);
      }
    }
    int32_t* dst = meta + p * kMetaInts;   // 4-byte aligned (all the ABI asks for)
#pragma unroll
    for (int j = 0; j < kMetaInts; ++j) dst[j] = (j == 0 || m[0] >= 0) ? m[j] : 0;
  }
  // 3. segments per request, prefix-summed into num_splits
  int64_t segs = 0;
  if (total > 0)
    for (int i = lo; i < hi; ++i) segs += segments(i, T);
  int64_t all_segs;
  int32_t r = static_cast<int32_t>(block_exclusive_scan<kT>(segs, s_scan, &all_segs));
  if (tid == 0) num_splits[0] = 0;
  for (int i = lo; i < hi; ++i) {
    if (total > 0) r += static_cast<int32_t>(segments(i, T));
    num_splits[i + 1] = r;
  }
}

}  // namespace mla
