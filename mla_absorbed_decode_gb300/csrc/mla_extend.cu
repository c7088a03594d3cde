// Chunked extend on the expanded path (MHA_CHUNKED_KV): "MLA 推理：两条计算路径与 FlashMLA",
// end of section "两条等价的路径" and exercise 3.  T new tokens of one request attend to its
// seqlen cached tokens (the new ones are the last T, causal); the cache is expanded chunk by
// chunk into per-head keys and values, each chunk is attended to on its own, and the chunks'
// results are merged by LSE, so the expanded context (~80 KB a token) never exists at once.
// Per chunk of the cache, two kernels:
//   1. mla_expand_kernel: Kx[t, h] = W_UK[h] c_t and Vx[t, h] = W_UV[h]^T c_t (128 values
//      each) for the chunk's tokens, a tcgen05 GEMM per (128-token tile, head): A = the
//      latent rows (two 64-token pages by TMA), B = W_UK[h] (K-major) and W_UV[h] (MN-major),
//      fp32 accumulators in TMEM, bf16 out.  Rows past the chunk are written as zeros.
//   2. mla_attend_kernel: per (128-query tile, head) a flash-attention loop over the chunk's
//      64-key tiles: S = [q_nope, q_pe] [Kx, k^R]^T (K = 192: Kx from the expansion, k^R
//      straight from the cache), online softmax in fp32 (one thread per query row, lazy
//      rescale of O at a 2^8 growth of the row maximum), O += P Vx, all MMAs on tcgen05 with
//      S and O in TMEM; the epilogue merges the chunk's (o, lse) into a running fp32
//      accumulator by log-sum-exp, and the last chunk writes the bf16 output and lse.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mla_kernels.h"
#include "mla_ptx.cuh"

namespace mla {

namespace {

constexpr uint64_t kExtTimeoutNs = 500ull * 1000 * 1000;

// Arrive on a named barrier without waiting (the producer side of a bar.arrive / bar.sync pair).
__device__ __forceinline__ void named_bar_arrive(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.arrive %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

__device__ __noinline__ bool ext_wait_slow(uint32_t bar, uint32_t parity, int* status) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > kExtTimeoutNs) {
      atomicCAS(status, 0, MLA_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}
// Bounded wait (0.5 s).  The phase is tested once before the clock is read: reading the
// global timer costs hundreds of cycles, which a wait that is already satisfied should not pay.
__device__ __forceinline__ bool ext_wait(uint32_t bar, uint32_t parity, int* status) {
  if (mbar_test(bar, parity)) return true;
  return ext_wait_slow(bar, parity, status);
}

// Stores 32 columns [c, c + 32) of the warp's 32 rows (one row per lane, values already
// bf16-packed as 16 words) through a 2 KiB transpose buffer: every store instruction
// writes 64 contiguous bytes of 8 rows.  rows_ok(x) says whether row x of the warp is kept.
template <typename F>
__device__ __forceinline__ void store_rows32(uint32_t stg, const uint32_t (&pk)[16], __nv_bfloat16* base,
                                             int64_t row_stride, int c, int lane, F rows_ok) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    st_shared_v4(stg + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4), make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]));
  __syncwarp();
  const int tq = lane & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int x = 8 * j + (lane >> 2);
    const uint4 u = ld_shared_v4(stg + x * 64 + ((tq ^ ((x >> 1) & 3)) << 4));
    if (rows_ok(x)) *reinterpret_cast<uint4*>(base + static_cast<int64_t>(x) * row_stride + c + 8 * tq) = u;
  }
  __syncwarp();
}

}  // namespace

// ---------------------------------------------------------------- expand --
constexpr int kExpStages = 2;
constexpr uint32_t kExpStage = 3 * 16384;   // latent chunk (A) + W_UK chunk (B, K-major) + W_UV chunk (B, MN-major)
constexpr uint32_t kExpSmem = kExpStages * kExpStage + 1024;

__global__ void __launch_bounds__(128, 2)
mla_expand_kernel(const __grid_constant__ CUtensorMap c_map, const __grid_constant__ CUtensorMap wk_map,
                  const __grid_constant__ CUtensorMap wv_map, const ExtendParams p) {
  extern __shared__ __align__(1024) uint8_t dyn_smem[];
  __shared__ uint64_t full[kExpStages], empty[kExpStages], acc_full;
  __shared__ uint32_t tmem_base_s;
  __shared__ int fail_s;
  const uint32_t smem = (smem_u32(dyn_smem) + 1023u) & ~1023u;
  const int tile = blockIdx.x, h = blockIdx.y;
  const int t0 = tile * 128;                    // first token of the tile, within the chunk
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kExpStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(&acc_full), 1);
    fail_s = 0;
    fence_mbar_init();
    prefetch_tensormap(&c_map);
    prefetch_tensormap(&wk_map);
    prefetch_tensormap(&wv_map);
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_base_s), 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  // The expansion of every chunk but the first reads only the cache and the weights, which
  // the kernels before it in the call do not write, and writes the Kx / Vx buffer that the
  // attention of the chunk before does not read (two buffers, alternating): it may run
  // beside that attention's last CTAs.  Its last CTA waits for that attention at its end
  // instead (the grid completes only after it), so that the attention after this kernel,
  // which waits for it, also finds the merged accumulator of the chunk before complete; the
  // other CTAs never wait, and leave their SMs as soon as they are done.
  if (!p.defer_wait) griddep_wait();
  griddep_launch_dependents();

  // the tile's (up to) two cache pages; a page past the chunk is not loaded (its rows are
  // never stored)
  const int pg0 = (p.c0 + t0) / kPageTokens;
  const bool two = t0 + 64 < p.n;
  int blk0 = __ldg(p.block_row + pg0), blk1 = two ? __ldg(p.block_row + pg0 + 1) : 0;
  if (blk0 < 0 || blk0 >= p.num_blocks || blk1 < 0 || blk1 >= p.num_blocks) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0, MLA_ERR_DEVICE_BOUNDS);
    blk0 = (blk0 < 0 || blk0 >= p.num_blocks) ? static_cast<int>(p.num_blocks) : blk0;   // TMA zero-fills it
    blk1 = (blk1 < 0 || blk1 >= p.num_blocks) ? static_cast<int>(p.num_blocks) : blk1;
  }
  const uint32_t stage_bytes = (two ? 2u : 1u) * 8192u + 2u * 16384u;
  int last_phase[kExpStages];
  for (int s = 0; s < kExpStages; ++s) last_phase[s] = -1;
  auto issue = [&](int kc) {   // latent dims [64 kc, 64 kc + 64)
    const int s = kc % kExpStages;
    const uint32_t st = smem + s * kExpStage;
    const uint32_t bar = smem_u32(&full[s]);
    mbar_arrive_expect_tx(bar, stage_bytes);
    tma_load_3d(st, &c_map, bar, 0, blk0 * kPageTokens, kc);
    if (two) tma_load_3d(st + 8192, &c_map, bar, 0, blk1 * kPageTokens, kc);
    tma_load_2d(st + 16384, &wk_map, bar, kc * 64, h * 128);                  // W_UK[h][0:128, 64 kc ..]
    tma_load_2d(st + 32768, &wv_map, bar, 0, h * kDimV + kc * 64);            // W_UV[h][64 kc .., 0:64]
    tma_load_2d(st + 32768 + 8192, &wv_map, bar, 64, h * kDimV + kc * 64);    // W_UV[h][64 kc .., 64:128]
    last_phase[s] = (kc / kExpStages) & 1;
  };
  if (threadIdx.x == 0)
    for (int kc = 0; kc < kExpStages; ++kc) issue(kc);
  if (warp == 0) {
    if (lane == 0)
      for (int kc = kExpStages; kc < kDimV / 64; ++kc) {
        if (!ext_wait(smem_u32(&empty[kc % kExpStages]), ((kc / kExpStages) - 1) & 1, p.status)) {
          fail_s = 1;
          break;
        }
        issue(kc);
      }
  } else if (warp == 1) {
    constexpr uint32_t id_k = idesc_bf16_f32(128, 128, 0, 0);   // B = W_UK[h] rows: K-major
    constexpr uint32_t id_v = idesc_bf16_f32(128, 128, 0, 1);   // B = W_UV[h] rows: MN-major
    bool ok = true;
    for (int kc = 0; kc < kDimV / 64; ++kc) {
      const int s = kc % kExpStages;
      ok = __all_sync(0xffffffffu, ext_wait(smem_u32(&full[s]), (kc / kExpStages) & 1, p.status));
      if (!ok) break;
      tc_fence_after();
      const uint32_t st = smem + s * kExpStage;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t a = smem_desc_sw128(st + kk * 32, 16, 1024);
        mma_bf16_ss_warp(tmem, a, smem_desc_sw128(st + 16384 + kk * 32, 16, 1024), id_k, (kc | kk) ? 1u : 0u);
        mma_bf16_ss_warp(tmem + 128, a, smem_desc_sw128(st + 32768 + kk * 2048, 8192, 1024), id_v,
                         (kc | kk) ? 1u : 0u);
      }
      mma_commit_warp(smem_u32(&empty[s]));
    }
    if (!ok && lane == 0) fail_s = 1;
    mma_commit_warp(smem_u32(&acc_full));
  }
  __syncthreads();
  const bool got = ext_wait(smem_u32(&acc_full), 0, p.status);
  tc_fence_after();
  const bool ok_all = got && !fail_s;
  // epilogue: row r of the tile -> Kx / Vx (zeros for rows past the chunk)
  const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  const uint32_t stg = smem + warp * 2048u;   // stage 0's latent part: idle now
  const int rw0 = t0 + warp * 32;
  for (int c = 0; c < 256; c += 32) {
    uint32_t v[32];
    tmem_ld32(tl + c, v);
    tmem_wait_ld();
    const bool in = rw0 + lane < p.n;
    uint32_t pk[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      pk[j] = in ? pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1])) : 0u;
    __nv_bfloat16* base = (c < 128 ? p.kx : p.vx) + (static_cast<int64_t>(h) * p.cap + rw0) * 128;   // [H][cap][128]
    store_rows32(stg, pk, base, 128, c & 127, lane,
                 [&](int x) { return ok_all && rw0 + x < p.cap; });
  }
  if (warp == 0 && lane == 0)   // loads in flight land before the CTA may exit
    for (int s = 0; s < kExpStages; ++s)
      if (last_phase[s] >= 0) ext_wait(smem_u32(&full[s]), static_cast<uint32_t>(last_phase[s]), p.status);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
  if (p.defer_wait && blockIdx.x == gridDim.x - 1 && blockIdx.y == gridDim.y - 1) griddep_wait();
}

// ---------------------------------------------------------------- attend --
// Two rings: a key stage (Kx tile, 2 x 8 KiB, + k^R tile, 8 KiB) is refilled as soon as its QK^T
// is done, a value stage (Vx tile, 2 x 8 KiB) after its PV, which comes a softmax later.  Key
// stages 4 and 5 reuse the query tile's shared memory once the query tile is in TMEM.
constexpr int kAttKStages = 6, kAttVStages = 4;
constexpr uint32_t kAttKStage = 24576, kAttVStage = 16384;
constexpr uint32_t kAttOffQ = 0;             // Q tile: 3 chunks of 64 dims x 128 rows (48 KiB)
constexpr uint32_t kAttOffStage = 49152;     // key stages 0..3, then the value stages
constexpr uint32_t kAttOffV = kAttOffStage + 4 * kAttKStage;
constexpr int kAttWG = 2;                      // softmax warpgroups: warpgroup g takes the key tiles k = g mod kAttWG
constexpr int kAttThreads = 128 + 128 * kAttWG + 32;   // warps 0-3, the softmax warpgroups, the value producer
// the epilogue's 2 KiB transpose buffer per softmax warp lies in the ring, idle once the last PV is done
constexpr uint32_t kAttOffEpi = kAttOffStage;
constexpr uint32_t kAttOffPm = kAttOffV + kAttVStages * kAttVStage;   // float [3][kAttWG][128]: exchange slots
constexpr uint32_t kAttSmem = kAttOffPm + 3 * kAttWG * 512 + 1024;
static_assert(kAttSmem <= 232448, "within one CTA's shared memory");
static_assert(kAttWG * 4 * 2048 <= 4 * kAttKStage, "the transpose buffers fit in the ring");
static_assert(kAttOffQ + (kAttKStages - 4) * kAttKStage <= kAttOffStage, "key stages 4.. fit in the query tile's memory");
__device__ __forceinline__ uint32_t att_kstage(uint32_t smem, int s) {
  return s < 4 ? smem + kAttOffStage + s * kAttKStage : smem + kAttOffQ + (s - 4) * kAttKStage;
}
// TMEM columns: O [0, 128), S (a 64-key buffer per softmax warpgroup), the query tile (A
// operand of QK^T: 192 dims, two per column, 96 columns), P (A operand of PV: 64 keys, a
// 32-column buffer per warpgroup).  With Q and P in TMEM both MMAs read only their B operand
// from shared memory.
constexpr uint32_t kAttTmemS = 128, kAttTmemQ = kAttTmemS + 64 * kAttWG, kAttTmemP = kAttTmemQ + 96;
static_assert(kAttTmemP + 32 * kAttWG <= 512, "O, S, Q and P fit in TMEM");
constexpr float kAttRebase = 8.0f;           // rebase the row maximum when it grows by more than 2^8

__global__ void __launch_bounds__(kAttThreads, 1)
mla_attend_kernel(const __grid_constant__ CUtensorMap qn_map, const __grid_constant__ CUtensorMap qp_map,
                  const __grid_constant__ CUtensorMap kx_map, const __grid_constant__ CUtensorMap vx_map,
                  const __grid_constant__ CUtensorMap kr_map, const ExtendParams p) {
  extern __shared__ __align__(1024) uint8_t dyn_smem[];
  __shared__ uint64_t kfull[kAttKStages], kempty[kAttKStages], vfull[kAttVStages], vempty[kAttVStages], q_full,
      q_tmem, s_full[kAttWG], s_empty[kAttWG], p_full[kAttWG], pv_done[kAttWG], drain;
  __shared__ uint32_t tmem_base_s;
  const uint32_t smem = (smem_u32(dyn_smem) + 1023u) & ~1023u;
  const int qt = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // keys of the chunk this query tile can see: positions c0 .. min(chunk end, last query's position)
  const int q_last = min(p.T, 128 * (qt + 1)) - 1;
  const int see_end = min(p.n, p.qpos0 + q_last + 1 - p.c0);          // keys [0, see_end) of the chunk
  const int ntiles = see_end > 0 ? (see_end + 63) / 64 : 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kAttKStages; ++s) {
      mbar_init(smem_u32(&kfull[s]), 1);
      mbar_init(smem_u32(&kempty[s]), 1);
    }
    for (int s = 0; s < kAttVStages; ++s) {
      mbar_init(smem_u32(&vfull[s]), 1);
      mbar_init(smem_u32(&vempty[s]), 1);
    }
    mbar_init(smem_u32(&q_full), 1);
    mbar_init(smem_u32(&q_tmem), 4 * kAttWG);   // every softmax warp, once the query tile is in TMEM
    for (int i = 0; i < kAttWG; ++i) {
      mbar_init(smem_u32(&s_full[i]), 1);
      mbar_init(smem_u32(&s_empty[i]), 4);   // the four warps of the warpgroup that owns buffer i
    }
    for (int i = 0; i < kAttWG; ++i) {
      mbar_init(smem_u32(&p_full[i]), 4);    // the four warps of the warpgroup that owns buffer i
      mbar_init(smem_u32(&pv_done[i]), 1);
    }
    mbar_init(smem_u32(&drain), 3);   // one commit from each MMA-issuing warp
    fence_mbar_init();
    prefetch_tensormap(&qn_map);
    prefetch_tensormap(&qp_map);
    prefetch_tensormap(&kx_map);
    prefetch_tensormap(&vx_map);
    prefetch_tensormap(&kr_map);
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_base_s), 512);   // O, S, Q, P (kAttTmem*)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {   // key producer: the query tile once, then the chunk's key tiles through the key ring
      const uint32_t qb = smem_u32(&q_full);
      mbar_arrive_expect_tx(qb, 3 * 16384);
      tma_load_3d(smem + kAttOffQ, &qn_map, qb, 0, h, 128 * qt);
      tma_load_3d(smem + kAttOffQ + 16384, &qn_map, qb, 64, h, 128 * qt);
      tma_load_3d(smem + kAttOffQ + 32768, &qp_map, qb, 0, h, 128 * qt);
      int kphase[kAttKStages];
      for (int s = 0; s < kAttKStages; ++s) kphase[s] = -1;
      for (int k = 0; k < ntiles; ++k) {
        const int s = k % kAttKStages;
        if (k >= kAttKStages && !ext_wait(smem_u32(&kempty[s]), ((k / kAttKStages) - 1) & 1, p.status)) break;
        if (k == 4) {   // stages 4.. are the query tile's memory: free once the softmax warps copied it to TMEM
          if (!ext_wait(smem_u32(&q_tmem), 0, p.status)) break;
          fence_proxy_async_smem();   // their generic-proxy reads before these async-proxy writes
        }
        int blk = __ldg(p.block_row + (p.c0 / kPageTokens) + k);
        if (blk < 0 || blk >= p.num_blocks) {
          atomicCAS(p.status, 0, MLA_ERR_DEVICE_BOUNDS);
          blk = static_cast<int>(p.num_blocks);   // out of range: the TMA fills the tile with zeros
        }
        const uint32_t st = att_kstage(smem, s);
        const uint32_t bar = smem_u32(&kfull[s]);
        mbar_arrive_expect_tx(bar, kAttKStage);
        tma_load_3d(st, &kx_map, bar, 0, 64 * k, h);
        tma_load_3d(st + 8192, &kx_map, bar, 64, 64 * k, h);
        tma_load_3d(st + 16384, &kr_map, bar, 0, blk * kPageTokens, kDimV / 64);   // k^R: cache dims 512..575
        kphase[s] = (k / kAttKStages) & 1;
      }
      ext_wait(qb, 0, p.status);   // loads in flight land before the CTA may exit
      for (int s = 0; s < kAttKStages; ++s)
        if (kphase[s] >= 0) ext_wait(smem_u32(&kfull[s]), static_cast<uint32_t>(kphase[s]), p.status);
    }
  } else if (warp == 1 || warp == 2) {   // QK^T issue (one elected lane), warp 1 the even tiles, warp 2 the odd
    // S = Q K^T of tile k into S buffer k % kAttWG, once the tile is loaded and the softmax has
    // read tile k - kAttWG out of that buffer.  QK^T (two warps) and PV (a third) are issued
    // apart: they share no accumulator, and each warp's waits and commits then overlap the
    // others' MMAs.
    constexpr uint32_t id_s = idesc_bf16_f32(128, 64, 0, 0);
    bool ok = __all_sync(0xffffffffu, ext_wait(smem_u32(&q_tmem), 0, p.status));
    tc_fence_after();
    for (int k = warp - 1; k < ntiles && ok; k += 2) {
      const int s = k % kAttKStages;
      const uint32_t sb = k % kAttWG;
      ok = __all_sync(0xffffffffu, ext_wait(smem_u32(&kfull[s]), (k / kAttKStages) & 1, p.status)) &&
           __all_sync(0xffffffffu, ext_wait(smem_u32(&s_empty[sb]), ((k / kAttWG) & 1) ^ 1, p.status));
      if (!ok) break;
      tc_fence_after();
      const uint64_t dk = smem_desc_sw128(att_kstage(smem, s), 16, 1024);
      const uint32_t sd = tmem + kAttTmemS + sb * 64;
#pragma unroll
      for (int c = 0; c < 3; ++c)   // q_nope . Kx (two 64-dim chunks), q_pe . k^R
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16_ts_warp(sd, tmem + kAttTmemQ + c * 32 + kk * 8, dk + ((c * 8192 + kk * 32) >> 4), id_s,
                           (c | kk) ? 1u : 0u);
      mma_commit_warp(smem_u32(&kempty[s]));
      mma_commit_warp(smem_u32(&s_full[sb]));
    }
    // this warp's MMAs are done before the CTA may free TMEM (also after a failure)
    mma_commit_warp(smem_u32(&drain));
    ext_wait(smem_u32(&drain), 0, p.status);
  } else if (warp == 3) {   // PV issue (one elected lane): O += P V for tile k, P from TMEM buffer k % kAttWG
    constexpr uint32_t id_o = idesc_bf16_f32(128, 128, 0, 1);
    bool ok = true;
    for (int k = 0; k < ntiles && ok; ++k) {
      const int s = k % kAttVStages;
      const int b = k % kAttWG;
      ok = __all_sync(0xffffffffu, ext_wait(smem_u32(&p_full[b]), (k / kAttWG) & 1, p.status)) &&
           __all_sync(0xffffffffu, ext_wait(smem_u32(&vfull[s]), (k / kAttVStages) & 1, p.status));
      if (!ok) break;
      tc_fence_after();
      const uint64_t dv = smem_desc_sw128(smem + kAttOffV + s * kAttVStage, 8192, 1024);
      const uint32_t pa = tmem + kAttTmemP + b * 32;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_bf16_ts_warp(tmem, pa + kk * 8, dv + (kk * 2048 >> 4), id_o, (k | kk) ? 1u : 0u);
      mma_commit_warp(smem_u32(&vempty[s]));
      mma_commit_warp(smem_u32(&pv_done[b]));
    }
    mma_commit_warp(smem_u32(&drain));
    ext_wait(smem_u32(&drain), 0, p.status);
  } else if (warp == 4 + 4 * kAttWG) {
    if (lane == 0) {   // value producer: the chunk's value tiles through the value ring
      int vphase[kAttVStages];
      for (int s = 0; s < kAttVStages; ++s) vphase[s] = -1;
      for (int k = 0; k < ntiles; ++k) {
        const int s = k % kAttVStages;
        if (k >= kAttVStages && !ext_wait(smem_u32(&vempty[s]), ((k / kAttVStages) - 1) & 1, p.status)) break;
        const uint32_t st = smem + kAttOffV + s * kAttVStage;
        const uint32_t bar = smem_u32(&vfull[s]);
        mbar_arrive_expect_tx(bar, kAttVStage);
        tma_load_3d(st, &vx_map, bar, 0, 64 * k, h);
        tma_load_3d(st + 8192, &vx_map, bar, 64, 64 * k, h);
        vphase[s] = (k / kAttVStages) & 1;
      }
      for (int s = 0; s < kAttVStages; ++s)   // loads in flight land before the CTA may exit
        if (vphase[s] >= 0) ext_wait(smem_u32(&vfull[s]), static_cast<uint32_t>(vphase[s]), p.status);
    }
  } else if (warp >= 4 && warp < 4 + 4 * kAttWG) {   // softmax and epilogue: kAttWG warpgroups, a thread per query row each
    // Warpgroup wg takes the key tiles k with k % kAttWG == wg whole (S buffer and P buffer wg),
    // so that the warpgroups run their tiles' softmax side by side.  The online softmax's one
    // serial dependency, the reference maximum, passes from tile k - 1 to tile k through a slot
    // per warpgroup and a named barrier per warpgroup (2 + g: "warpgroup g has published"),
    // taken bar.arrive by the publisher and bar.sync by the next warpgroup.  Every tile's barrier operations are
    // executed whatever happened before (a failed wait only skips the work), so neither side
    // can be left waiting.  The reference maximum only moves when a tile's maximum exceeds it
    // by more than 2^kAttRebase; the warpgroup whose tile moves it rescales O (after the PV of
    // tile k - 1), and each warpgroup rescales its own partial row sum when it sees it move.
    constexpr uint32_t kST = 128 * kAttWG;           // softmax threads
    const int t = threadIdx.x - 128, wg = t >> 7, r = t & 127, wq = r >> 5;
    const int q = 128 * qt + r;                      // query row within the request
    const int qpos = p.qpos0 + q;                    // its position
    const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    // slot j of warpgroup g: j = 0 the reference maximum it published last, j = 1 / 2 its
    // reference and row sum after the loop
    const auto pm = [&](int j, int g) { return smem + kAttOffPm + ((j * kAttWG + g) * 128 + r) * 4; };
    float m = -INFINITY, l = 0.f;   // this warpgroup's reference maximum (log2 units) and row sum over its tiles
    // the query tile into TMEM: row r's 192 dims (three 128-byte swizzled chunks) as 96
    // columns of bf16 pairs, chunk c by warpgroup c % kAttWG
    bool ok = __all_sync(0xffffffffu, ext_wait(smem_u32(&q_full), 0, p.status));
    if (ok) {
      for (int c = wg; c < 3; c += kAttWG) {
        uint32_t v[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 x = ld_shared_v4(smem + kAttOffQ + c * 16384 + r * 128 + ((u ^ (r & 7)) << 4));
          v[4 * u] = x.x, v[4 * u + 1] = x.y, v[4 * u + 2] = x.z, v[4 * u + 3] = x.w;
        }
        tmem_st32(tl + kAttTmemQ + c * 32, v);
      }
      tmem_wait_st();
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&q_tmem));   // arrives even after a failure: the MMA warp's wait ends
    const uint32_t sb = wg;                          // this warpgroup's S and P buffers
    const int prev = (wg + kAttWG - 1) % kAttWG;     // the warpgroup of the tile before
    for (int k = wg; k < ntiles; k += kAttWG) {
      const uint32_t ph = (k / kAttWG) & 1;          // phase of this warpgroup's buffers for tile k
      ok = __all_sync(0xffffffffu, ok && ext_wait(smem_u32(&s_full[sb]), ph, p.status));
      float x[64];
      if (ok) {
        tc_fence_after();
        tmem_ld32(tl + kAttTmemS + sb * 64, *reinterpret_cast<uint32_t(*)[32]>(x));
        tmem_ld32(tl + kAttTmemS + sb * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(x + 32));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s_empty[sb]));
      }
      // the keys a row sees form a prefix of the tile: inside the chunk and at or before
      // this query's position
      const int t0 = p.c0 + 64 * k;
      const int nvis = (ok && q < p.T) ? min(p.n - 64 * k, qpos - t0 + 1) : 0;
      if (nvis < 64) {
#pragma unroll
        for (int j = 0; j < 64; ++j) x[j] = j < nvis ? x[j] : -INFINITY;
      }
      float mx[32];   // the row maximum by a tree
#pragma unroll
      for (int j = 0; j < 32; ++j) mx[j] = fmaxf(x[2 * j], x[2 * j + 1]);
#pragma unroll
      for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
        for (int j = 0; j < w; ++j) mx[j] = fmaxf(mx[j], mx[j + w]);
      // the reference maximum after tile k - 1, from the warpgroup before
      float m_in = -INFINITY;
      if (k > 0) {
        named_bar_sync(2 + prev, 256);
        m_in = ld_shared_f32(pm(0, prev));
      }
      // softmax_scale > 0, so the scaled maximum is the scaled raw maximum
      const float cand = mx[0] * p.scale_log2;
      const float m_k = cand > m_in + kAttRebase ? cand : m_in;   // the reference for tile k
      if (k + 1 < ntiles) {
        asm volatile("st.shared.f32 [%0], %1;" :: "r"(pm(0, wg)), "f"(m_k) : "memory");
        named_bar_arrive(2 + wg, 256);
      }
      if (m_k != m) {   // m_k > m: this warpgroup's row sum moves to the new reference (0 when m = -inf)
        l *= fast_exp2(m - m_k);
        m = m_k;
      }
      // A row whose reference this tile moves has O (every earlier tile, once the PV of tile
      // k - 1 is done; the MMAs complete in order) scaled by 2^(m_in - m_k); with m_in = -inf
      // every earlier P was 0, and so is O.  The decision is per row, but the wait and the
      // TMEM loads and stores are warp-wide: if any row of the warp moves, the whole warp
      // rescales, by 1 where its row does not.
      const bool moves = m_k != m_in && k > 0 && m_in != -INFINITY;
      if (ok && __any_sync(0xffffffffu, moves)) {
        const float alpha = moves ? fast_exp2(m_in - m_k) : 1.f;
        ok = __all_sync(0xffffffffu,
                        ext_wait(smem_u32(&pv_done[(k - 1) % kAttWG]), ((k - 1) / kAttWG) & 1, p.status));
        if (ok) {
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 128; c += 32) {
            uint32_t v[32];
            tmem_ld32(tl + c, v);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
            tmem_st32(tl + c, v);
          }
          tmem_wait_st();
        }
      }
      // P buffer sb is free once the PV of tile k - kAttWG (which read it) is done
      if (ok && k >= kAttWG) ok = __all_sync(0xffffffffu, ext_wait(smem_u32(&pv_done[sb]), ph ^ 1, p.status));
      if (ok) {
        const float neg_m = (m_k == -INFINITY) ? 0.f : -m_k;
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {   // P of the tile's 64 keys as bf16 pairs, 32 keys at a time
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float a = fast_exp2(fmaf(x[32 * hf + 2 * e], p.scale_log2, neg_m));   // 2^-inf = +0
            const float b = fast_exp2(fmaf(x[32 * hf + 2 * e + 1], p.scale_log2, neg_m));
            ps[e & 3] += a + b;
            w[e] = pack_bf16x2(a, b);
          }
          tmem_st16(tl + kAttTmemP + sb * 32 + 16 * hf, w);
        }
        tmem_wait_st();
        l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&p_full[sb]));
      }
    }
    if (ok && ntiles > 0)
      ok = __all_sync(0xffffffffu, ext_wait(smem_u32(&pv_done[(ntiles - 1) % kAttWG]), ((ntiles - 1) / kAttWG) & 1,
                                            p.status));
    // the row sums at the largest reference, which is O's (the barrier also settles whether
    // every warp finished)
    asm volatile("st.shared.f32 [%0], %1;" :: "r"(pm(1, wg)), "f"(m) : "memory");
    asm volatile("st.shared.f32 [%0], %1;" :: "r"(pm(2, wg)), "f"(l) : "memory");
    ok = !named_bar_or(1, kST, !ok);
    {
      float m_f = m;
#pragma unroll
      for (int g = 0; g < kAttWG; ++g) m_f = fmaxf(m_f, ld_shared_f32(pm(1, g)));
      if (m_f != -INFINITY) {
        float l_f = 0.f;
#pragma unroll
        for (int g = 0; g < kAttWG; ++g) l_f += ld_shared_f32(pm(2, g)) * fast_exp2(ld_shared_f32(pm(1, g)) - m_f);
        l = l_f;
      }
      m = m_f;
    }
    tc_fence_after();
    // epilogue: the chunk's o = O / l and lse, merged into the running accumulator by LSE;
    // warpgroup wg writes the 32-column chunks c = wg mod kAttWG of O
    const bool row_ok = ok && q < p.T;
    const float lse_c = (l > 0.f) ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
    const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
    const int64_t row = static_cast<int64_t>(q) * p.H + h;
    float lse_a = -INFINITY;
    if (row_ok && !p.first) lse_a = p.acc_lse[row];
    const float M = fmaxf(lse_a, lse_c);
    const float wa = (M == -INFINITY || lse_a == -INFINITY) ? 0.f : expf(lse_a - M);
    const float wc = (M == -INFINITY || lse_c == -INFINITY) ? 0.f : expf(lse_c - M);
    const float z = wa + wc;
    const float ca = z > 0.f ? wa / z : 0.f, cc = z > 0.f ? wc * inv_l / z : 0.f;
    const float lse_new = z > 0.f ? M + logf(z) : -INFINITY;
    const uint32_t stg = smem + kAttOffEpi + (wg * 4 + wq) * 2048u;
    const int qw0 = 128 * qt + wq * 32;
    for (int c = 32 * wg; c < 128; c += 32 * kAttWG) {
      uint32_t v[32];
      if (ntiles > 0) {
        tmem_ld32(tl + c, v);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0u;
      }
      float o[32];
      const float4* a4 = reinterpret_cast<const float4*>(p.acc_o + row * 128 + c);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 a = (row_ok && ca > 0.f) ? a4[j] : make_float4(0.f, 0.f, 0.f, 0.f);
        o[4 * j + 0] = ca * a.x + cc * __uint_as_float(v[4 * j + 0]);
        o[4 * j + 1] = ca * a.y + cc * __uint_as_float(v[4 * j + 1]);
        o[4 * j + 2] = ca * a.z + cc * __uint_as_float(v[4 * j + 2]);
        o[4 * j + 3] = ca * a.w + cc * __uint_as_float(v[4 * j + 3]);
      }
      if (p.last) {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(o[2 * j], o[2 * j + 1]);
        store_rows32(stg, pk, p.out + (static_cast<int64_t>(qw0) * p.H + h) * 128, static_cast<int64_t>(p.H) * 128, c,
                     lane, [&](int x) { return ok && qw0 + x < p.T; });
      } else if (row_ok) {
        float4* d4 = reinterpret_cast<float4*>(p.acc_o + row * 128 + c);
#pragma unroll
        for (int j = 0; j < 8; ++j) d4[j] = make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
      }
    }
    if (row_ok && wg == 0) {
      if (p.last) p.lse[row] = lse_new;
      else p.acc_lse[row] = lse_new;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t extend_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(mla_expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kExpSmem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(mla_attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kAttSmem));
}

cudaError_t launch_extend_chunk(const ExtendMaps& maps, const ExtendParams& p, int buf, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  {
    const cudaLaunchConfig_t cfg = pdl_config(dim3(static_cast<unsigned>((p.n + 127) / 128), static_cast<unsigned>(p.H)),
                                              dim3(128), kExpSmem, stream, attr);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, mla_expand_kernel, maps.c, maps.wk, maps.wv, p);
    if (e != cudaSuccess) return e;
  }
  const cudaLaunchConfig_t cfg = pdl_config(dim3(static_cast<unsigned>((p.T + 127) / 128), static_cast<unsigned>(p.H)),
                                            dim3(kAttThreads), kAttSmem, stream, attr);
  return cudaLaunchKernelEx(&cfg, mla_attend_kernel, maps.qn, maps.qp, maps.kx[buf], maps.vx[buf], maps.kr, p);
}

}  // namespace mla
