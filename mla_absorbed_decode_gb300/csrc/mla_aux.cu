// Split-KV tile scheduler, LSE combine of split partials, and the W_UK / W_UV
// per-head projections on tcgen05.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mla_kernels.h"
#include "mla_ptx.cuh"
#include "mla_rope.cuh"
#include "mla_schedule.cuh"

namespace mla {

// --------------------------------------------------------------- schedule --
__global__ void __launch_bounds__(kScheduleThreads) mla_schedule_kernel(const int32_t* seqlens, int B, int num_parts,
                                                                        int fixed_cost, int hbm_parts, int split_cost,
                                                                        int32_t* meta, int32_t* num_splits) {
  extern __shared__ int64_t sched_c[];                                      // C[0..B]
  int32_t* sched_nb = reinterpret_cast<int32_t*>(sched_c + B + 1);         // nb[0..B)
  __shared__ int64_t s_scan[kScheduleThreads / 32 + 1];
  griddep_wait();
  griddep_launch_dependents();
  schedule_body<kScheduleThreads>(seqlens, B, num_parts, fixed_cost, hbm_parts, split_cost, meta, num_splits, sched_c,
                                  sched_nb, s_scan);
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
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = pdl_config(dim3(1), dim3(kScheduleThreads), smem, stream, attr);
  return cudaLaunchKernelEx(&cfg, mla_schedule_kernel, seqlens, B, num_parts, fixed_cost, hbm_parts, split_cost, meta,
                            num_splits);
}

// ---------------------------------------------------------------- combine --
// Merge the fp32 partials of split requests by log-sum-exp (same page: "合并各段
// 的部分结果"; the chunk merge of MHA_CHUNKED_KV is the same rule):
//   lse = ln sum_k exp(lse_k),   out = sum_k exp(lse_k - lse) o_k.
// One warp per row, 16 output values per lane.  Requests with one segment were
// written by the decode kernel; requests with none get out = 0, lse = -inf.
__global__ void __launch_bounds__(128)
mla_combine_kernel(const float* o_part, const float* lse_part, const int32_t* num_splits, int B, int rows,
                   int max_splits, __nv_bfloat16* out, float* lse, int* status) {
  griddep_wait();
  griddep_launch_dependents();
  const int b = blockIdx.x;
  const int g = blockIdx.y * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B || g >= rows) return;
  const int s0 = num_splits[b];
  const int n = num_splits[b + 1] - s0;
  if (n == 1) return;
  if (s0 < 0 || n < 0 || s0 + n > max_splits) {   // offsets that do not fit the workspace: reported, not read
    if (lane == 0) atomicCAS(status, 0, MLA_ERR_DEVICE_BOUNDS);
    return;
  }
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
    // two partials per pass, their loads issued together (a long merge is latency-
    // bound otherwise); a partial with weight 0 is never multiplied in
    for (int k0 = 0; k0 < n; k0 += 2) {
      const bool two = k0 + 1 < n;
      const int64_t r0 = static_cast<int64_t>(s0 + k0) * rows + g;
      const int64_t r1 = two ? r0 + rows : r0;
      const float l0 = lse_part[r0], l1 = lse_part[r1];
      const float w0 = (l0 == -INFINITY) ? 0.f : expf(l0 - m);
      const float w1 = (!two || l1 == -INFINITY) ? 0.f : expf(l1 - m);
      const float4* p0 = reinterpret_cast<const float4*>(o_part + r0 * kDimV + lane * 16);
      const float4* p1 = reinterpret_cast<const float4*>(o_part + r1 * kDimV + lane * 16);
      float4 v0[4], v1[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v0[j] = p0[j];
      if (two) {
#pragma unroll
        for (int j = 0; j < 4; ++j) v1[j] = p1[j];
      }
      z += w0;
      if (w0 != 0.f) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[4 * j + 0] += w0 * v0[j].x;
          acc[4 * j + 1] += w0 * v0[j].y;
          acc[4 * j + 2] += w0 * v0[j].z;
          acc[4 * j + 3] += w0 * v0[j].w;
        }
      }
      z += w1;
      if (w1 != 0.f) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[4 * j + 0] += w1 * v1[j].x;
          acc[4 * j + 1] += w1 * v1[j].y;
          acc[4 * j + 2] += w1 * v1[j].z;
          acc[4 * j + 3] += w1 * v1[j].w;
        }
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
// NT = 128): "DeepSeekV2之MLA" 4.5, the bmm calls with w_kc and w_vc.
// K is walked in chunks of 64 through a ring of STAGES shared-memory stages; a
// stage holds the A chunk (128 tokens x 64, K-major, one 3-D TMA box over
// [K, H, N]) and the W chunk (64 rows of W[h] x NT columns, N contiguous, so an
// MN-major B operand: NT / 64 2-D boxes over [H*K, N_total]).  The accumulator is
// in TMEM; one thread issues TMA, one warp the MMAs, and all 128 threads run the
// epilogue (one token row each), with the TMEM load of the next 32 columns in
// flight while the previous ones are stored.
template <int K, int NT, int STAGES>
__host__ __device__ constexpr uint32_t bmm_stage_bytes() {
  return 16384u + static_cast<uint32_t>(NT) * 128u;
}
template <int K, int NT, int STAGES>
uint32_t bmm_smem_bytes() {
  return STAGES * bmm_stage_bytes<K, NT, STAGES>() + 1024;
}

__device__ __noinline__ bool bmm_wait_slow(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > 500000000ull) return false;
  }
  return true;
}
// Bounded wait (0.5 s).  The phase is tested once before the clock is read: reading the
// global timer costs hundreds of cycles, which a wait that is already satisfied should not pay.
__device__ __forceinline__ bool bmm_wait(uint32_t bar, uint32_t parity) {
  if (mbar_test(bar, parity)) return true;
  return bmm_wait_slow(bar, parity);
}

// TMA store of a 3-D box from shared memory (completion tracked by the bulk-group helpers).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
               :: "l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(x), "r"(y), "r"(z) : "memory");
}

template <int K, int NT, int STAGES>
__global__ void __launch_bounds__(128, 1)
mla_bmm_kernel(const __grid_constant__ CUtensorMap a_map, const __grid_constant__ CUtensorMap w_map,
               const __grid_constant__ CUtensorMap o_map, const BmmParams p) {
  static_assert(K % 64 == 0 && NT % 64 == 0 && NT >= 64 && NT <= 256 && STAGES >= 1, "tile shape");
  constexpr int KC = K / 64;
  constexpr uint32_t kSB = bmm_stage_bytes<K, NT, STAGES>();
  constexpr uint32_t kTmemCols = NT;
  constexpr int kNX = (K == 128 ? 512 : 128) / NT;   // column tiles per head
  extern __shared__ __align__(1024) uint8_t dyn_smem[];
  __shared__ uint64_t full[STAGES], empty[STAGES], acc_full;
  __shared__ uint32_t tmem_base_s;
  __shared__ int fail_s;
  const uint32_t smem = (smem_u32(dyn_smem) + 1023u) & ~1023u;
  // the grid is flat: column tile fastest, then head, then 128-token tile; with a
  // schedule to compute, one CTA past the tiles does that and nothing else
  const int tile = static_cast<int>(blockIdx.x);
  if (p.sched_meta != nullptr && tile == kNX * p.H * ((p.N + 127) / 128)) {
    __shared__ int64_t sched_scan[128 / 32 + 1];
    int64_t* sched_c = reinterpret_cast<int64_t*>(dyn_smem + (smem - smem_u32(dyn_smem)));
    griddep_wait();   // the lengths may come from the previous kernel
    griddep_launch_dependents();
    schedule_body<128>(p.sched_seqlens, p.sched_B, p.sched_parts, p.sched_fixed, p.sched_hbm, p.sched_split,
                       p.sched_meta, p.sched_meta + kMetaInts * p.sched_parts, sched_c,
                       reinterpret_cast<int32_t*>(sched_c + p.sched_B + 1), sched_scan);
    return;
  }
  const int n0 = (tile % kNX) * NT, h = (tile / kNX) % p.H, m0 = (tile / (kNX * p.H)) * 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(&acc_full), 1);
    fail_s = 0;
    fence_mbar_init();
    prefetch_tensormap(&a_map);
    prefetch_tensormap(&w_map);
    // this head's weight matrix (K x 512 or 512 x 128 bf16, 128 KiB) into L2 while the
    // previous kernel of the stream may still run, for the chunks past the ring (one CTA
    // per head issues it)
    if (p.w != nullptr && n0 == 0 && m0 == 0)
      prefetch_l2(p.w + static_cast<int64_t>(h) * K * (K == 128 ? 512 : 128), static_cast<uint32_t>(K) * (K == 128 ? 512 : 128) * 2);
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_base_s), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  // producer (warp 0, lane 0): K chunks through the ring.  The weights are not written by
  // the previous kernel of the stream, so the chunks that fit the ring at once have their
  // weight parts issued before griddepcontrol.wait, overlapping that kernel's tail; the
  // activations (A) follow once it is done.
  int last_phase[STAGES];
  for (int s = 0; s < STAGES; ++s) last_phase[s] = -1;
  auto issue_w = [&](int c) {   // expects the whole stage, loads its weight part
    const int s = c % STAGES;
    const uint32_t st = smem + s * kSB;
    const uint32_t bar = smem_u32(&full[s]);
    mbar_arrive_expect_tx(bar, kSB);
#pragma unroll
    for (int j = 0; j < NT / 64; ++j) tma_load_2d(st + 16384 + j * 8192, &w_map, bar, n0 + j * 64, h * K + c * 64);
    last_phase[s] = (c / STAGES) & 1;
  };
  auto issue_a = [&](int c) {
    const int s = c % STAGES;
    tma_load_3d(smem + s * kSB, &a_map, smem_u32(&full[s]), c * 64, h, m0);
  };
  constexpr int kFirst = KC < STAGES ? KC : STAGES;
  if (warp == 0 && lane == 0)
    for (int c = 0; c < kFirst; ++c) issue_w(c);
  griddep_wait();
  griddep_launch_dependents();
  if (warp == 0 && lane == 0)
    for (int c = 0; c < kFirst; ++c) issue_a(c);

  const int n = m0 + threadIdx.x;
  // the RoPE part of the decode query is copied by the first column tile; it is
  // loaded (and rotated) while the tiles are in flight
  const bool copy_pe = n0 == 0 && p.pe != nullptr && n < p.N;
  uint4 pe[8];
  if (copy_pe) {
    const uint4* src = reinterpret_cast<const uint4*>(p.pe + static_cast<int64_t>(n) * p.pe_row_stride + h * 64);
#pragma unroll
    for (int j = 0; j < 8; ++j) pe[j] = __ldg(src + j);
    if (p.positions != nullptr) rope_row(pe, __ldg(p.positions + n), p);
  }

  if (warp == 0) {
    if (lane == 0) {   // the rest of K, each chunk once the MMAs have freed its stage
      for (int c = kFirst; c < KC; ++c) {
        if (!bmm_wait(smem_u32(&empty[c % STAGES]), ((c / STAGES) - 1) & 1)) {
          fail_s = 1;
          break;
        }
        issue_w(c);
        issue_a(c);
      }
    }
  } else if (warp == 1) {   // MMA issue: the whole warp waits, one elected lane issues
    constexpr uint32_t idesc = idesc_bf16_f32(128, NT, 0, 1);
    bool ok = true;
    for (int c = 0; c < KC; ++c) {
      const int s = c % STAGES;
      ok = __all_sync(0xffffffffu, bmm_wait(smem_u32(&full[s]), (c / STAGES) & 1));
      if (!ok) break;
      tc_fence_after();
      const uint32_t st = smem + s * kSB;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t a = smem_desc_sw128(st + kk * 32, 16, 1024);
        const uint64_t w = smem_desc_sw128(st + 16384 + kk * 2048, 8192, 1024);
        mma_bf16_ss_warp(tmem, a, w, idesc, (c > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit_warp(smem_u32(&empty[s]));
    }
    if (!ok && lane == 0) fail_s = 1;
    mma_commit_warp(smem_u32(&acc_full));   // arrives once every MMA issued so far is done
  }
  __syncthreads();
  const bool got = bmm_wait(smem_u32(&acc_full), 0);
  tc_fence_after();
  if ((!got || fail_s) && threadIdx.x == 0) atomicCAS(p.status, 0, MLA_ERR_TIMEOUT);
  const bool store = got && !fail_s && n < p.N;
  __nv_bfloat16* dst = p.out + static_cast<int64_t>(n) * p.out_row_stride + static_cast<int64_t>(h) * p.out_head_stride + n0;
  const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  // The stores go out by TMA: warp w stages its 32 token rows as one 32-row x 64-column tile
  // per 64 output columns (the 128-byte swizzle of the output map: row r's 16-byte unit u at
  // r * 128 + ((u ^ (r & 7)) * 16), so that each store instruction of the warp covers all 32
  // banks), in the idle ring, and one lane stores each tile; rows past N are clipped by the
  // map.  A warp whose rows all lie past N does nothing.
  const int nw0 = m0 + warp * 32;
  const bool ok_all = got && !fail_s;
  const uint32_t stg = smem + warp * (NT / 64) * 4096u;
  if (ok_all && nw0 < p.N) {
#pragma unroll 1
    for (int g = 0; g < NT / 64; ++g) {
      uint32_t va[32], vb[32];
      tmem_ld32(tl + 64 * g, va);
      tmem_ld32(tl + 64 * g + 32, vb);
      tmem_wait_ld();
      const uint32_t row = stg + g * 4096u + lane * 128u;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t* v = u < 4 ? va + 8 * u : vb + 8 * (u - 4);
        uint4 x;
        x.x = pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1]));
        x.y = pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3]));
        x.z = pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5]));
        x.w = pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7]));
        st_shared_v4(row + ((u ^ (lane & 7)) << 4), x);
      }
    }
    fence_proxy_async_smem();   // the staged tiles are visible to the TMA (async proxy)
    __syncwarp();
    if (lane == 0) {
      for (int g = 0; g < NT / 64; ++g) tma_store_3d(&o_map, stg + g * 4096u, n0 + 64 * g, h, nw0);
      bulk_commit_group();
      bulk_wait_group_read<0>();   // the tiles are read before the CTA may exit
    }
    __syncwarp();
  }
  if (store && copy_pe) {
    uint4* d4 = reinterpret_cast<uint4*>(dst + 512);
#pragma unroll
    for (int j = 0; j < 8; ++j) d4[j] = pe[j];
  }
  if (warp == 0 && lane == 0)   // loads in flight land before the CTA may exit
    for (int s = 0; s < STAGES; ++s)
      if (last_phase[s] >= 0) bmm_wait(smem_u32(&full[s]), static_cast<uint32_t>(last_phase[s]));
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// absorb: K = 128 -> two 256-column tiles of 512; un-absorb: K = 512 -> one 128-column tile
#define MLA_BMM_ABSORB 128, 256, 2
#define MLA_BMM_UNABSORB 512, 128, 6

cudaError_t bmm_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(mla_bmm_kernel<MLA_BMM_ABSORB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bmm_smem_bytes<MLA_BMM_ABSORB>()));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(mla_bmm_kernel<MLA_BMM_UNABSORB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bmm_smem_bytes<MLA_BMM_UNABSORB>()));
}

cudaError_t launch_bmm(bool absorb, const CUtensorMap& a_map, const CUtensorMap& w_map, const CUtensorMap& o_map,
                       const BmmParams& p, cudaStream_t stream) {
  const int64_t mt = (p.N + 127) / 128;
  cudaLaunchAttribute attr[1];
  if (absorb) {
    if (p.sched_meta != nullptr &&
        (p.sched_B < 1 || p.sched_B > kAbsorbPlanMaxB || p.sched_parts < 1 ||
         sizeof(int64_t) * (p.sched_B + 1) + sizeof(int32_t) * p.sched_B + 1024 > bmm_smem_bytes<MLA_BMM_ABSORB>()))
      return cudaErrorInvalidValue;
    const int64_t ctas = (512 / 256) * static_cast<int64_t>(p.H) * mt + (p.sched_meta != nullptr ? 1 : 0);
    if (ctas > 0x7fffffff) return cudaErrorInvalidValue;
    const cudaLaunchConfig_t cfg = pdl_config(dim3(static_cast<unsigned>(ctas)), dim3(128),
                                              bmm_smem_bytes<MLA_BMM_ABSORB>(), stream, attr);
    return cudaLaunchKernelEx(&cfg, mla_bmm_kernel<MLA_BMM_ABSORB>, a_map, w_map, o_map, p);
  }
  if (p.sched_meta != nullptr) return cudaErrorInvalidValue;
  const int64_t ctas = (128 / 128) * static_cast<int64_t>(p.H) * mt;
  if (ctas > 0x7fffffff) return cudaErrorInvalidValue;
  const cudaLaunchConfig_t cfg = pdl_config(dim3(static_cast<unsigned>(ctas)), dim3(128),
                                            bmm_smem_bytes<MLA_BMM_UNABSORB>(), stream, attr);
  return cudaLaunchKernelEx(&cfg, mla_bmm_kernel<MLA_BMM_UNABSORB>, a_map, w_map, o_map, p);
}


cudaError_t launch_combine(const float* o_part, const float* lse_part, const int32_t* num_splits, int B, int rows,
                           int max_splits, __nv_bfloat16* out, float* lse, int* status, cudaStream_t stream) {
  // The decode kernel never signals its dependents early, so the combine's CTAs are
  // placed only once the whole decode grid is done (spread over every SM) and the
  // programmatic launch just hides the launch latency.  An early signal would let them
  // pile onto the few SMs that the decode frees first, where the merge of long
  // requests then runs alone.
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg =
      pdl_config(dim3(static_cast<unsigned>(B), static_cast<unsigned>((rows + 3) / 4), 1), dim3(128), 0, stream, attr);
  return cudaLaunchKernelEx(&cfg, mla_combine_kernel, o_part, lse_part, num_splits, B, rows, max_splits, out, lse,
                            status);
}

}  // namespace mla
