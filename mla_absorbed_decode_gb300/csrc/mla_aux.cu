// Split-KV tile scheduler, LSE combine of split partials, and the W_UK / W_UV
// per-head projections on tcgen05.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mla_kernels.h"
#include "mla_ptx.cuh"

namespace mla {

// --------------------------------------------------------------- schedule --
// get_mla_metadata's role ("MLA 推理：两条计算路径与 FlashMLA", FlashMLA paragraph):
// from the sequence lengths alone, decide which KV pages each part (cluster)
// processes; at most `hbm_parts` parts are used, since that many already keep HBM
// busy, unless using all parts is estimated to be faster even with the splits it
// causes (`split_cost` pages per extra segment).  One CTA.  Every request is laid out on a line of cost positions: F set-up
// positions, then one position per page; request b occupies [C[b], C[b+1]).  The
// line is cut into P_eff equal pieces of T = ceil(C[B] / P_eff) positions, part p
// taking the pages whose positions lie in [p T, (p + 1) T).  The costs are
// prefix-summed by all threads; each part then finds its first and last page with
// two binary searches, independently of the other parts.
__global__ void __launch_bounds__(kScheduleThreads) mla_schedule_kernel(const int32_t* seqlens, int B, int num_parts,
                                                                        int fixed_cost, int hbm_parts, int split_cost,
                                                                        int32_t* meta, int32_t* num_splits) {
  extern __shared__ int64_t sched_c[];                                      // C[0..B]
  int32_t* sched_nb = reinterpret_cast<int32_t*>(sched_c + B + 1);         // nb[0..B)
  __shared__ int64_t s_part[kScheduleThreads];
  const int tid = threadIdx.x;
  const int64_t F = fixed_cost;
  const int chunk = (B + kScheduleThreads - 1) / kScheduleThreads;
  const int lo = min(B, tid * chunk), hi = min(B, lo + chunk);
  // 1. page counts, per-thread sums of the costs, block-wide exclusive scan, C
  int64_t sum = 0;
  for (int i = lo; i < hi; ++i) {
    const int L = seqlens[i];
    const int nb = L > 0 ? (L + kPageTokens - 1) / kPageTokens : 0;
    sched_nb[i] = nb;
    sum += nb > 0 ? nb + F : 0;
  }
  s_part[tid] = sum;
  __syncthreads();
  if (tid == 0) {
    int64_t run = 0;
    for (int j = 0; j < kScheduleThreads; ++j) {
      const int64_t v = s_part[j];
      s_part[j] = run;
      run += v;
    }
    sched_c[0] = 0;
  }
  __syncthreads();
  int64_t run = s_part[tid];
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
      __syncthreads();
      s_part[tid] = extra;
      __syncthreads();
      if (tid == 0) {
        int64_t e = 0;
        for (int j = 0; j < kScheduleThreads; ++j) e += s_part[j];
        s_part[0] = e;
      }
      __syncthreads();
      const int64_t est = Tc + static_cast<int64_t>(split_cost) * ((s_part[0] + pe - 1) / pe);
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
  for (int p = tid; p < num_parts; p += kScheduleThreads) {
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
  int32_t segs = 0;
  if (total > 0)
    for (int i = lo; i < hi; ++i) segs += static_cast<int32_t>(segments(i, T));
  __syncthreads();
  s_part[tid] = segs;
  __syncthreads();
  if (tid == 0) {
    int64_t r = 0;
    for (int j = 0; j < kScheduleThreads; ++j) {
      const int64_t v = s_part[j];
      s_part[j] = r;
      r += v;
    }
    num_splits[0] = 0;
  }
  __syncthreads();
  int32_t r = static_cast<int32_t>(s_part[tid]);
  for (int i = lo; i < hi; ++i) {
    if (total > 0) r += static_cast<int32_t>(segments(i, T));
    num_splits[i + 1] = r;
  }
}

cudaError_t launch_schedule(const int32_t* seqlens, int B, int num_parts, int fixed_cost, int hbm_parts,
                            int split_cost, int32_t* meta, int32_t* num_splits, cudaStream_t stream) {
  if (B < 1 || B > kScheduleMaxB) return cudaErrorInvalidValue;
  const size_t smem = sizeof(int64_t) * (static_cast<size_t>(B) + 1) + sizeof(int32_t) * static_cast<size_t>(B);
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(mla_schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  mla_schedule_kernel<<<1, kScheduleThreads, smem, stream>>>(seqlens, B, num_parts, fixed_cost, hbm_parts,
                                                              split_cost, meta, num_splits);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- combine --
// Merge the fp32 partials of split requests by log-sum-exp (same page: "合并各段
// 的部分结果"; the chunk merge of MHA_CHUNKED_KV is the same rule):
//   lse = ln sum_k exp(lse_k),   out = sum_k exp(lse_k - lse) o_k.
// One warp per row, 16 output values per lane.  Requests with one segment were
// written by the decode kernel; requests with none get out = 0, lse = -inf.
__global__ void __launch_bounds__(128)
mla_combine_kernel(const float* o_part, const float* lse_part, const int32_t* num_splits, int B, int rows,
                   __nv_bfloat16* out, float* lse) {
  const int b = blockIdx.x;
  const int g = blockIdx.y * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B || g >= rows) return;
  const int s0 = num_splits[b];
  const int n = num_splits[b + 1] - s0;
  if (n == 1) return;
  __nv_bfloat16* orow = out + (static_cast<int64_t>(b) * rows + g) * kDimV + lane * 16;
  if (n == 0) {
    const uint4 z = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(orow)[0] = z;
    reinterpret_cast<uint4*>(orow)[1] = z;
    if (lane == 0) lse[static_cast<int64_t>(b) * rows + g] = -INFINITY;
    return;
  }
  float m = -INFINITY;
  for (int k = lane; k < n; k += 32) m = fmaxf(m, lse_part[static_cast<int64_t>(s0 + k) * rows + g]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float acc[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j] = 0.f;
  float z = 0.f;
  if (m != -INFINITY) {
    for (int k = 0; k < n; ++k) {
      const float lk = lse_part[static_cast<int64_t>(s0 + k) * rows + g];
      const float wk = (lk == -INFINITY) ? 0.f : expf(lk - m);
      z += wk;
      if (wk == 0.f) continue;
      const float4* src = reinterpret_cast<const float4*>(o_part + (static_cast<int64_t>(s0 + k) * rows + g) * kDimV +
                                                          lane * 16);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 v = src[j];
        acc[4 * j + 0] += wk * v.x;
        acc[4 * j + 1] += wk * v.y;
        acc[4 * j + 2] += wk * v.z;
        acc[4 * j + 3] += wk * v.w;
      }
    }
  }
  const float inv = z > 0.f ? 1.f / z : 0.f;
  uint4 u[2];
  uint32_t* w = reinterpret_cast<uint32_t*>(u);
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = pack_bf16x2(acc[2 * j] * inv, acc[2 * j + 1] * inv);
  reinterpret_cast<uint4*>(orow)[0] = u[0];
  reinterpret_cast<uint4*>(orow)[1] = u[1];
  if (lane == 0) lse[static_cast<int64_t>(b) * rows + g] = z > 0.f ? m + logf(z) : -INFINITY;
}

// -------------------------------------------------------------------- bmm --
// out[n, h, n0 : n0+NT] = A[n, h, 0:K] @ W[h][0:K, n0 : n0+NT]  for a tile of
// 128 tokens n, one head h and one NT-wide column tile.  Used for the W_UK
// absorption (K = 128, NT = 256 of 512) and the W_UV un-absorption (K = 512,
// NT = 64 of 128): "DeepSeekV2之MLA" 4.5, the bmm calls with w_kc and w_vc.
// A (K-major) arrives by a 3-D TMA [K, H, N] in 64-wide swizzled boxes; W[h]
// (N contiguous, so an MN-major B operand) by a 2-D TMA over [H*K, N_total].
// The accumulator is in TMEM; one thread issues TMA and MMA, 128 threads run
// the epilogue (one token row each).
template <int K, int NT>
uint32_t bmm_smem_bytes() {
  return 128 * K * 2 + K * NT * 2 + 1024;
}

template <int K, int NT>
__global__ void __launch_bounds__(128, 1)
mla_bmm_kernel(const __grid_constant__ CUtensorMap a_map, const __grid_constant__ CUtensorMap w_map,
               const BmmParams p) {
  static_assert(K % 64 == 0 && NT % 64 == 0 && NT <= 256, "tile shape");
  constexpr uint32_t kABytes = 128 * K * 2;         // K/64 boxes of [128 rows x 128 B]
  constexpr uint32_t kWChunk = K * 128;             // one 64-column chunk of W[h]: K rows x 128 B
  constexpr int kWBoxRows = K > 256 ? 256 : K;
  constexpr uint32_t kTmemCols = NT < 32 ? 32 : NT;
  extern __shared__ __align__(1024) uint8_t dyn_smem[];
  __shared__ uint64_t bar_tma, bar_mma;
  __shared__ uint32_t tmem_base_s;
  const uint32_t smem = (smem_u32(dyn_smem) + 1023u) & ~1023u;
  const uint32_t sA = smem, sW = smem + kABytes;
  const int n0 = blockIdx.x * NT, h = blockIdx.y, m0 = blockIdx.z * 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar_tma), 1);
    mbar_init(smem_u32(&bar_mma), 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_base_s), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  __shared__ int ok_s;
  if (threadIdx.x == 0) {
    ok_s = 0;
    mbar_arrive_expect_tx(smem_u32(&bar_tma), kABytes + (NT / 64) * kWChunk);
#pragma unroll 1
    for (int c = 0; c < K / 64; ++c) tma_load_3d(sA + c * 16384, &a_map, smem_u32(&bar_tma), c * 64, h, m0);
#pragma unroll 1
    for (int j = 0; j < NT / 64; ++j)
#pragma unroll 1
      for (int r0 = 0; r0 < K; r0 += kWBoxRows)
        tma_load_2d(sW + j * kWChunk + r0 * 128, &w_map, smem_u32(&bar_tma), n0 + j * 64, h * K + r0);
  }
  if (warp == 0) {   // the whole warp waits; one elected lane issues the MMAs
    const uint64_t t0 = global_timer_ns();
    bool got = true;
    while (!mbar_test(smem_u32(&bar_tma), 0)) {
      if (global_timer_ns() - t0 > 500000000ull) { got = false; break; }
    }
    got = __all_sync(0xffffffffu, got);
    if (got) {
      tc_fence_after();
      constexpr uint32_t idesc = idesc_bf16_f32(128, NT, 0, 1);
#pragma unroll
      for (int kk = 0; kk < K / 16; ++kk) {
        const uint64_t a = smem_desc_sw128(sA + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
        const uint64_t w = smem_desc_sw128(sW + kk * 2048, kWChunk, 1024);
        mma_bf16_ss_warp(tmem, a, w, idesc, kk > 0 ? 1u : 0u);
      }
      mma_commit_warp(smem_u32(&bar_mma));
      if (lane == 0) ok_s = 1;
    } else if (lane == 0) {
      atomicCAS(p.status, 0, MLA_ERR_TIMEOUT);
      mbar_arrive(smem_u32(&bar_mma));   // release the epilogue without MMAs in flight
    }
  }
  {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_test(smem_u32(&bar_mma), 0)) {
      if (global_timer_ns() - t0 > 500000000ull) break;
    }
  }
  tc_fence_after();
  __syncthreads();
  const int n = m0 + threadIdx.x;
  const bool store = ok_s && n < p.N;
  __nv_bfloat16* dst = p.out + static_cast<int64_t>(n) * p.out_row_stride + static_cast<int64_t>(h) * p.out_head_stride + n0;
  const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
  for (int c = 0; c < NT; c += 32) {
    uint32_t v[32];
    tmem_ld32(tl + c, v);
    tmem_wait_ld();
    if (store) {
      uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint4 u;
        u.x = pack_bf16x2(__uint_as_float(v[8 * j + 0]), __uint_as_float(v[8 * j + 1]));
        u.y = pack_bf16x2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3]));
        u.z = pack_bf16x2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5]));
        u.w = pack_bf16x2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7]));
        d4[j] = u;
      }
    }
  }
  if (store && blockIdx.x == 0 && p.pe != nullptr) {   // RoPE part of the decode query
    const uint4* src = reinterpret_cast<const uint4*>(p.pe + static_cast<int64_t>(n) * p.pe_row_stride + h * 64);
    uint4* d4 = reinterpret_cast<uint4*>(dst + 512);
#pragma unroll
    for (int j = 0; j < 8; ++j) d4[j] = __ldg(src + j);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

cudaError_t bmm_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(mla_bmm_kernel<128, 256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bmm_smem_bytes<128, 256>()));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(mla_bmm_kernel<512, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bmm_smem_bytes<512, 64>()));
}

cudaError_t launch_bmm(bool absorb, const CUtensorMap& a_map, const CUtensorMap& w_map, const BmmParams& p,
                       cudaStream_t stream) {
  const unsigned mt = static_cast<unsigned>((p.N + 127) / 128);
  if (absorb) {
    mla_bmm_kernel<128, 256><<<dim3(2, p.H, mt), 128, bmm_smem_bytes<128, 256>(), stream>>>(a_map, w_map, p);
  } else {
    mla_bmm_kernel<512, 64><<<dim3(2, p.H, mt), 128, bmm_smem_bytes<512, 64>(), stream>>>(a_map, w_map, p);
  }
  return cudaGetLastError();
}


cudaError_t launch_combine(const float* o_part, const float* lse_part, const int32_t* num_splits, int B, int rows,
                           __nv_bfloat16* out, float* lse, cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>(B), static_cast<unsigned>((rows + 3) / 4), 1);
  mla_combine_kernel<<<grid, 128, 0, stream>>>(o_part, lse_part, num_splits, B, rows, out, lse);
  return cudaGetLastError();
}

}  // namespace mla
