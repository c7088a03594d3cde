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

__device__ __forceinline__ bool ext_wait(uint32_t bar, uint32_t parity, int* status) {   // bounded
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > kExtTimeoutNs) {
      atomicCAS(status, 0, MLA_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
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
  griddep_wait();
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
}

// ---------------------------------------------------------------- attend --
constexpr int kAttStages = 3;
constexpr uint32_t kAttStage = 40960;        // Kx tile (2 x 8 KiB) + k^R tile (8 KiB) + Vx tile (2 x 8 KiB)
constexpr uint32_t kAttOffQ = 0;             // Q tile: 3 chunks of 64 dims x 128 rows (48 KiB)
constexpr uint32_t kAttOffStage = 49152;
constexpr uint32_t kAttOffEpi = kAttOffStage + kAttStages * kAttStage;   // 8 x 2 KiB transpose buffers
constexpr uint32_t kAttOffPm = kAttOffEpi + 16384;   // float [3][2][128]: row maxima by tile parity, then row sums
constexpr uint32_t kAttSmem = kAttOffPm + 3072 + 1024;
// TMEM columns: O [0, 128), S (two 64-key buffers) [128, 256), the query tile (A operand of
// QK^T: 192 dims, two per column) [256, 352), P (A operand of PV: 64 keys, two buffers)
// [352, 416).  With Q and P in TMEM both MMAs read only their B operand from shared memory.
constexpr uint32_t kAttTmemS = 128, kAttTmemQ = 256, kAttTmemP = 352;
constexpr float kAttRebase = 8.0f;           // rebase the row maximum when it grows by more than 2^8

__global__ void __launch_bounds__(384, 1)
mla_attend_kernel(const __grid_constant__ CUtensorMap qn_map, const __grid_constant__ CUtensorMap qp_map,
                  const __grid_constant__ CUtensorMap kx_map, const __grid_constant__ CUtensorMap vx_map,
                  const __grid_constant__ CUtensorMap kr_map, const ExtendParams p) {
  extern __shared__ __align__(1024) uint8_t dyn_smem[];
  __shared__ uint64_t full[kAttStages], empty[kAttStages], q_full, q_tmem, s_full[2], s_empty[2], p_full[2],
      pv_done[2], drain;
  __shared__ uint32_t tmem_base_s;
  const uint32_t smem = (smem_u32(dyn_smem) + 1023u) & ~1023u;
  const int qt = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // keys of the chunk this query tile can see: positions c0 .. min(chunk end, last query's position)
  const int q_last = min(p.T, 128 * (qt + 1)) - 1;
  const int see_end = min(p.n, p.qpos0 + q_last + 1 - p.c0);          // keys [0, see_end) of the chunk
  const int ntiles = see_end > 0 ? (see_end + 63) / 64 : 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kAttStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(&q_full), 1);
    mbar_init(smem_u32(&q_tmem), 8);   // the eight softmax warps, once the query tile is in TMEM
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s_full[i]), 1);
      mbar_init(smem_u32(&s_empty[i]), 8);   // the eight softmax warps
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&p_full[i]), 8);    // the eight softmax warps
      mbar_init(smem_u32(&pv_done[i]), 1);
    }
    mbar_init(smem_u32(&drain), 1);
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
    if (lane == 0) {   // producer: the query tile once, then the chunk's key tiles through the ring
      const uint32_t qb = smem_u32(&q_full);
      mbar_arrive_expect_tx(qb, 3 * 16384);
      tma_load_3d(smem + kAttOffQ, &qn_map, qb, 0, h, 128 * qt);
      tma_load_3d(smem + kAttOffQ + 16384, &qn_map, qb, 64, h, 128 * qt);
      tma_load_3d(smem + kAttOffQ + 32768, &qp_map, qb, 0, h, 128 * qt);
      int issued_phase[kAttStages];
      for (int s = 0; s < kAttStages; ++s) issued_phase[s] = -1;
      bool ok = true;
      for (int k = 0; k < ntiles && ok; ++k) {
        const int s = k % kAttStages;
        if (k >= kAttStages && !ext_wait(smem_u32(&empty[s]), ((k / kAttStages) - 1) & 1, p.status)) {
          ok = false;
          break;
        }
        int blk = __ldg(p.block_row + (p.c0 / kPageTokens) + k);
        if (blk < 0 || blk >= p.num_blocks) {
          atomicCAS(p.status, 0, MLA_ERR_DEVICE_BOUNDS);
          blk = static_cast<int>(p.num_blocks);   // out of range: the TMA fills the tile with zeros
        }
        const uint32_t st = smem + kAttOffStage + s * kAttStage;
        const uint32_t bar = smem_u32(&full[s]);
        mbar_arrive_expect_tx(bar, kAttStage);
        tma_load_3d(st, &kx_map, bar, 0, 64 * k, h);
        tma_load_3d(st + 8192, &kx_map, bar, 64, 64 * k, h);
        tma_load_3d(st + 16384, &kr_map, bar, 0, blk * kPageTokens, kDimV / 64);   // k^R: cache dims 512..575
        tma_load_3d(st + 24576, &vx_map, bar, 0, 64 * k, h);
        tma_load_3d(st + 32768, &vx_map, bar, 64, 64 * k, h);
        issued_phase[s] = (k / kAttStages) & 1;
      }
      ext_wait(qb, 0, p.status);   // loads in flight land before the CTA may exit
      for (int s = 0; s < kAttStages; ++s)
        if (issued_phase[s] >= 0) ext_wait(smem_u32(&full[s]), static_cast<uint32_t>(issued_phase[s]), p.status);
    }
  } else if (warp == 1) {   // MMA issue (one elected lane), QK^T of tile k ahead of PV of tile k - 1
    constexpr uint32_t id_s = idesc_bf16_f32(128, 64, 0, 0);
    constexpr uint32_t id_o = idesc_bf16_f32(128, 128, 0, 1);
    bool ok = __all_sync(0xffffffffu, ext_wait(smem_u32(&q_tmem), 0, p.status));
    tc_fence_after();
    auto pv = [&](int k) {   // O += P V for tile k, P from TMEM buffer k % 2
      if (!__all_sync(0xffffffffu, ext_wait(smem_u32(&p_full[k & 1]), (k >> 1) & 1, p.status))) return false;
      tc_fence_after();
      const uint32_t st = smem + kAttOffStage + (k % kAttStages) * kAttStage;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_bf16_ts_warp(tmem, tmem + kAttTmemP + (k & 1) * 32 + kk * 8,
                         smem_desc_sw128(st + 24576 + kk * 2048, 8192, 1024), id_o, (k | kk) ? 1u : 0u);
      mma_commit_warp(smem_u32(&empty[k % kAttStages]));
      mma_commit_warp(smem_u32(&pv_done[k & 1]));
      return true;
    };
    for (int k = 0; k < ntiles && ok; ++k) {
      const int s = k % kAttStages;
      const uint32_t sb = k & 1;
      ok = __all_sync(0xffffffffu, ext_wait(smem_u32(&full[s]), (k / kAttStages) & 1, p.status)) &&
           __all_sync(0xffffffffu, ext_wait(smem_u32(&s_empty[sb]), ((k >> 1) & 1) ^ 1, p.status));
      if (!ok) break;
      tc_fence_after();
      const uint32_t st = smem + kAttOffStage + s * kAttStage;
#pragma unroll
      for (int c = 0; c < 3; ++c)   // q_nope . Kx (two 64-dim chunks), q_pe . k^R
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16_ts_warp(tmem + kAttTmemS + sb * 64, tmem + kAttTmemQ + c * 32 + kk * 8,
                           smem_desc_sw128(st + c * 8192 + kk * 32, 16, 1024), id_s, (c | kk) ? 1u : 0u);
      mma_commit_warp(smem_u32(&s_full[sb]));
      if (k > 0 && !pv(k - 1)) ok = false;
    }
    if (ok && ntiles > 0) pv(ntiles - 1);
    // every MMA issued so far is done before the CTA may free TMEM (also after a failure)
    mma_commit_warp(smem_u32(&drain));
    ext_wait(smem_u32(&drain), 0, p.status);
  } else if (warp >= 4) {   // softmax and epilogue: two warpgroups, one thread per query row each
    // warpgroup wg takes keys [32 wg, 32 wg + 32) of every tile and O columns [64 wg, 64 wg + 64);
    // the two agree on the row maximum (and so on every rebase) through pm[][] and named
    // barrier 1, and add their partial row sums at the end
    const int t = threadIdx.x - 128, wg = t >> 7, r = t & 127, wq = r >> 5;
    const int q = 128 * qt + r;                      // query row within the request
    const int qpos = p.qpos0 + q;                    // its position
    const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    // exchange slot j of this warpgroup / of the other one; j = tile parity in the loop, 2 after
    // it (with one barrier per tile a warpgroup writes slot k % 2 again only after the other
    // has passed the next barrier, i.e. after it read that slot)
    const auto pm_mine = [&](int j) { return smem + kAttOffPm + ((j * 2 + wg) * 128 + r) * 4; };
    const auto pm_other = [&](int j) { return smem + kAttOffPm + ((j * 2 + 1 - wg) * 128 + r) * 4; };
    float m = -INFINITY, l = 0.f;                    // reference maximum (log2 units), this half's row sum
    // the query tile into TMEM: row r's 192 dims (three 128-byte swizzled chunks) as 96
    // columns of bf16 pairs (warpgroup 0: q_nope, warpgroup 1: q_pe)
    bool ok = __all_sync(0xffffffffu, ext_wait(smem_u32(&q_full), 0, p.status));
    if (ok) {
      for (int c = wg == 0 ? 0 : 2; c < (wg == 0 ? 2 : 3); ++c) {
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
    // Every exit from the loop is taken by all eight warps together, after a barrier that
    // folds in each warp's wait results (a warp leaving alone would strand the others there).
    for (int k = 0; k < ntiles; ++k) {
      const uint32_t sb = k & 1;
      const bool got = __all_sync(0xffffffffu, ok && ext_wait(smem_u32(&s_full[sb]), (k >> 1) & 1, p.status));
      float x[32];
      if (got) {
        tc_fence_after();
        tmem_ld32(tl + kAttTmemS + sb * 64 + wg * 32, *reinterpret_cast<uint32_t(*)[32]>(x));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s_empty[sb]));
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = -INFINITY;
      }
      // the keys a row sees form a prefix of the tile: inside the chunk and at or before
      // this query's position
      const int t0 = p.c0 + 64 * k;
      const int nvis = q < p.T ? min(p.n - 64 * k, qpos - t0 + 1) : 0;
      const int nvalid = nvis - 32 * wg;                // of this warpgroup's 32 keys
      if (nvalid < 32) {
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = j < nvalid ? x[j] : -INFINITY;
      }
      float rmax = x[0];
#pragma unroll
      for (int j = 1; j < 32; ++j) rmax = fmaxf(rmax, x[j]);
      asm volatile("st.shared.f32 [%0], %1;" :: "r"(pm_mine(k & 1)), "f"(rmax) : "memory");
      // P buffer k % 2 is free once the PV of tile k - 2 (which read it) is done
      bool go = got;
      if (go && k > 1 && !ext_wait(smem_u32(&pv_done[k & 1]), ((k >> 1) & 1) ^ 1, p.status)) go = false;
      // one barrier both exchanges the row maxima and makes the abort decision uniform
      if (named_bar_or(1, 256, !go)) { ok = false; break; }
      // softmax_scale > 0, so the scaled maximum is the scaled raw maximum
      const float m_new = fmaxf(m, fmaxf(rmax, ld_shared_f32(pm_other(k & 1))) * p.scale_log2);
      if (m_new > m + kAttRebase) {   // rebase: O and l scale by 2^(m - m_new) (0 when m = -inf)
        const float alpha = fast_exp2(m - m_new);
        l *= alpha;
        // O holds every earlier tile once the PV of tile k - 1 is done (the MMAs complete in order);
        // a failed wait is carried to the next barrier (or the one after the loop)
        if (k > 0 && !__all_sync(0xffffffffu, ext_wait(smem_u32(&pv_done[(k - 1) & 1]), ((k - 1) >> 1) & 1,
                                                        p.status))) {
          ok = false;
        }
        if (k > 0 && ok) {
          tc_fence_after();
#pragma unroll 1
          for (int c = 64 * wg; c < 64 * wg + 64; c += 32) {
            uint32_t v[32];
            tmem_ld32(tl + c, v);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
            tmem_st32(tl + c, v);
          }
          tmem_wait_st();
        }
        m = m_new;
      }
      const float neg_m = (m == -INFINITY) ? 0.f : -m;
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t w[16];   // P of this half's 32 keys as bf16 pairs (2^x of -inf is +0)
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float a = fast_exp2(fmaf(x[2 * e], p.scale_log2, neg_m));
        const float b = fast_exp2(fmaf(x[2 * e + 1], p.scale_log2, neg_m));
        ps[e & 3] += a + b;
        w[e] = pack_bf16x2(a, b);
      }
      tmem_st16(tl + kAttTmemP + (k & 1) * 32 + wg * 16, w);
      tmem_wait_st();
      l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&p_full[k & 1]));
    }
    if (ok && ntiles > 0)
      ok = __all_sync(0xffffffffu, ext_wait(smem_u32(&pv_done[(ntiles - 1) & 1]), ((ntiles - 1) >> 1) & 1, p.status));
    // the row sum over both halves (the barrier also settles whether every warp finished)
    asm volatile("st.shared.f32 [%0], %1;" :: "r"(pm_mine(2)), "f"(l) : "memory");
    ok = !named_bar_or(1, 256, !ok);
    l += ld_shared_f32(pm_other(2));
    tc_fence_after();
    // epilogue: the chunk's o = O / l and lse, merged into the running accumulator by LSE;
    // warpgroup wg writes O columns [64 wg, 64 wg + 64)
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
    for (int c = 64 * wg; c < 64 * wg + 64; c += 32) {
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

cudaError_t launch_extend_chunk(const ExtendMaps& maps, const ExtendParams& p, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  {
    const cudaLaunchConfig_t cfg = pdl_config(dim3(static_cast<unsigned>((p.n + 127) / 128), static_cast<unsigned>(p.H)),
                                              dim3(128), kExpSmem, stream, attr);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, mla_expand_kernel, maps.c, maps.wk, maps.wv, p);
    if (e != cudaSuccess) return e;
  }
  const cudaLaunchConfig_t cfg = pdl_config(dim3(static_cast<unsigned>((p.T + 127) / 128), static_cast<unsigned>(p.H)),
                                            dim3(384), kAttSmem, stream, attr);
  return cudaLaunchKernelEx(&cfg, mla_attend_kernel, maps.qn, maps.qp, maps.kx, maps.vx, maps.kr, p);
}

}  // namespace mla
