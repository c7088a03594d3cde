// W_UK / W_UV projections on FP8 tensor cores (the FP8 branch of the absorption):
//     x_val, x_scale = input_to_float8(x);   y = bmm_fp8(x_val, w, x_scale, w_scale) -> bf16
// ("SGLang v0.3 MLA / torch.compile" handbook page, the weight-absorption code walk-
// through: q_nope before W_UK, the attention output before W_UV, one scale per operand).
//
// The activation's scale is per tensor: it maps the largest |x| of the whole [N, H, K]
// tensor onto 448, E4M3's largest finite value.  That needs every CTA to know the global
// maximum before it quantizes its tile, so a call runs two kernels on the stream:
//   1. mla_amax_kernel: kAmaxParts CTAs each write the maximum |x| of their share of x;
//   2. mla_bmm_fp8_kernel: each CTA reduces those partial maxima (a few hundred bytes),
//      loads its bf16 x tile by TMA, quantizes it on chip into the MMA operand layout,
//      multiplies it with the E4M3 weight tile (TMA, stored transposed: K contiguous) on
//      kind::f8f6f4 tensor cores with fp32 accumulation in TMEM, and writes
//      acc * x_scale * w_scale in bf16.
// The quantization takes the same float32 steps as the oracle (inv = 448 / amax,
// code = e4m3_rn_satfinite(x * inv)), so both reach the same codes.  The weight tile is
// loaded before griddepcontrol.wait (the weights are not written by the previous kernel of
// the stream), so its HBM read overlaps the tail of that kernel; x and the partial maxima
// are read after it.  The bf16 result leaves by TMA stores of swizzled 32 x 64 tiles.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mla_kernels.h"
#include "mla_ptx.cuh"
#include "mla_rope.cuh"
#include "mla_schedule.cuh"

namespace mla {

namespace {
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
}  // namespace

// ---------------------------------------------------------- amax partials --
// partials[blockIdx.x] = max |x| over the grid-stride share of x of CTA blockIdx.x <
// kAmaxParts, x viewed as `rows` rows of `row_units` 16-byte units (8 bf16 values) at
// `row_stride` elements apart.  With sched.sched_meta set, CTA kAmaxParts computes the
// split schedule instead (mla_decode_metadata's output), its prefix sums in the launch's
// dynamic shared memory.
__global__ void __launch_bounds__(256) mla_amax_kernel(const __nv_bfloat16* x, int64_t rows, int64_t row_units,
                                                       int64_t row_stride, float* partials,
                                                       const BmmParams sched) {
  if (sched.sched_meta != nullptr && blockIdx.x == kAmaxParts) {
    extern __shared__ int64_t amax_sched_c[];
    __shared__ int64_t amax_scan[256 / 32 + 1];
    griddep_wait();   // the lengths may come from the previous kernel
    griddep_launch_dependents();
    schedule_body<256>(sched.sched_seqlens, sched.sched_B, sched.sched_parts, sched.sched_fixed, sched.sched_hbm,
                       sched.sched_split, sched.sched_meta, sched.sched_meta + kMetaInts * sched.sched_parts,
                       amax_sched_c, reinterpret_cast<int32_t*>(amax_sched_c + sched.sched_B + 1), amax_scan);
    return;
  }
  griddep_wait();
  griddep_launch_dependents();
  const int64_t total = rows * row_units;
  float m = 0.f;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < total;
       u += static_cast<int64_t>(kAmaxParts) * blockDim.x) {
    const int64_t r = u / row_units, c = u - r * row_units;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + r * row_stride) + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float wmax[8];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = wmax[0];
    for (int i = 1; i < static_cast<int>(blockDim.x >> 5); ++i) b = fmaxf(b, wmax[i]);
    partials[blockIdx.x] = b;
  }
}

// ------------------------------------------------------------- FP8 bmm --
// A CTA computes out[n, h, n0 : n0 + NT] for 128 tokens n (one M tile), one head h and one
// NT-wide column tile.  Shared memory (from a 1024-byte aligned base):
//   W codes: K / 128 chunks of NT rows x 128 codes (K-major B operand, 128-byte swizzle);
//   A codes: K / 128 chunks of 128 token rows x 128 codes (K-major A operand, same swizzle);
//   x ring:  bf16 x chunks of 64 values x 128 rows (16 KiB TMA boxes, 128-byte swizzle),
//            reused as the epilogue's transpose buffers once the codes are written.
template <int K, int NT>
struct Fp8BmmShape {
  static constexpr int kXChunks = K / 64;
  static constexpr int kXStages = kXChunks < 4 ? kXChunks : 4;
  static constexpr int kCodeChunks = K / 128;
  static constexpr uint32_t kWBytes = static_cast<uint32_t>(kCodeChunks) * NT * 128;
  static constexpr uint32_t kABytes = static_cast<uint32_t>(kCodeChunks) * 128 * 128;
  static constexpr uint32_t kOffW = 0;
  static constexpr uint32_t kOffA = kWBytes;
  static constexpr uint32_t kOffX = kOffA + kABytes;
  static constexpr uint32_t kSmem = kOffX + kXStages * 16384u + 1024u;   // + alignment slack
  static_assert(K % 128 == 0 && NT % 16 == 0 && NT >= 32 && NT <= 256, "tile shape");
};

// TMA store of a 3-D box from shared memory (completion tracked by the bulk-group helpers).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
               :: "l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(x), "r"(y), "r"(z) : "memory");
}

template <int K, int NT>
__global__ void __launch_bounds__(128, 1)
mla_bmm_fp8_kernel(const __grid_constant__ CUtensorMap x_map, const __grid_constant__ CUtensorMap w_map,
                   const __grid_constant__ CUtensorMap o_map, const BmmFp8Params p) {
  using S = Fp8BmmShape<K, NT>;
  extern __shared__ __align__(1024) uint8_t dyn_smem[];
  __shared__ uint64_t w_full, x_full[S::kXStages], x_empty[S::kXStages], acc_full;
  __shared__ uint32_t tmem_base_s;
  __shared__ float red[4];
  __shared__ int fail_s;
  const uint32_t smem = (smem_u32(dyn_smem) + 1023u) & ~1023u;
  const int n0 = blockIdx.x * NT, h = blockIdx.y, m0 = blockIdx.z * 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = threadIdx.x;   // this thread's token row in the tile (its TMEM lane)
  const BmmParams& b = p.base;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&w_full), 1);
    for (int s = 0; s < S::kXStages; ++s) {
      mbar_init(smem_u32(&x_full[s]), 1);
      mbar_init(smem_u32(&x_empty[s]), 128);
    }
    mbar_init(smem_u32(&acc_full), 1);
    fail_s = 0;
    fence_mbar_init();
    prefetch_tensormap(&x_map);
    prefetch_tensormap(&w_map);
    prefetch_tensormap(&o_map);
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_base_s), NT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  // producer: the whole weight tile (while the previous kernel may still run), then the
  // first x chunks
  bool issued_w = false;
  if (threadIdx.x == 0) {
    const uint32_t bar = smem_u32(&w_full);
    mbar_arrive_expect_tx(bar, S::kWBytes);
#pragma unroll
    for (int cc = 0; cc < S::kCodeChunks; ++cc)
      tma_load_2d(smem + S::kOffW + cc * (NT * 128u), &w_map, bar, cc * 128, h * p.J + n0);
    issued_w = true;
  }
  griddep_wait();
  griddep_launch_dependents();
  int x_issued = 0;
  auto issue_x = [&](int c) {
    const int s = c % S::kXStages;
    const uint32_t bar = smem_u32(&x_full[s]);
    mbar_arrive_expect_tx(bar, 16384);
    tma_load_3d(smem + S::kOffX + s * 16384u, &x_map, bar, c * 64, h, m0);
  };
  if (threadIdx.x == 0) {
    for (int c = 0; c < S::kXStages; ++c) issue_x(c);
    x_issued = S::kXStages;
  }

  // the per-tensor scale of x from the partial maxima (kAmaxParts = blockDim.x values)
  static_assert(kAmaxParts == 128, "one partial maximum per thread");
  float m = __ldg(p.partials + threadIdx.x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  const float amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;       // 448 / amax, float32
  const float x_scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;   // amax / 448, float32
  const float out_scale = x_scale * p.w_scale;

  // every thread quantizes its own row: x chunk c (64 values) -> codes 64c .. 64c + 63
  bool ok = true;
  for (int c = 0; c < S::kXChunks; ++c) {
    const int s = c % S::kXStages;
    const uint32_t ph = (c / S::kXStages) & 1;
    if (!bmm_wait(smem_u32(&x_full[s]), ph)) {
      ok = false;
      break;
    }
    const uint32_t xrow = smem + S::kOffX + s * 16384u + r * 128u;
    const uint32_t arow = smem + S::kOffA + (c >> 1) * 16384u + r * 128u;
#pragma unroll
    for (int t = 0; t < 4; ++t) {   // two bf16 units (16 values) -> one 16-byte code unit
      const uint4 v0 = ld_shared_v4(xrow + (((2 * t) ^ (r & 7)) << 4));
      const uint4 v1 = ld_shared_v4(xrow + (((2 * t + 1) ^ (r & 7)) << 4));
      const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      uint32_t cw[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {   // 4 codes per 32-bit word
        const uint32_t lo = cvt_e4m3x2(__fmul_rn(bf16_lo(w[2 * j]), inv), __fmul_rn(bf16_hi(w[2 * j]), inv));
        const uint32_t hi = cvt_e4m3x2(__fmul_rn(bf16_lo(w[2 * j + 1]), inv), __fmul_rn(bf16_hi(w[2 * j + 1]), inv));
        cw[j] = lo | (hi << 16);
      }
      const int unit = (c & 1) * 4 + t;
      st_shared_v4(arow + ((unit ^ (r & 7)) << 4), make_uint4(cw[0], cw[1], cw[2], cw[3]));
    }
    mbar_arrive(smem_u32(&x_empty[s]));
    if (threadIdx.x == 0 && x_issued < S::kXChunks) {   // refill this stage once every row is converted
      if (!bmm_wait(smem_u32(&x_empty[s]), ph)) {
        ok = false;
        break;
      }
      issue_x(x_issued++);
    }
  }
  if (!ok) fail_s = 1;
  fence_proxy_async_smem();   // the codes were written by the generic proxy; the MMAs read them
  __syncthreads();

  if (warp == 1) {   // MMA issue: the whole warp waits, one elected lane issues
    constexpr uint32_t idesc = idesc_e4m3_f32(128, NT, 0, 0);
    bool mok = (fail_s == 0) && __all_sync(0xffffffffu, bmm_wait(smem_u32(&w_full), 0));
    if (mok) {
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < S::kCodeChunks; ++cc)
#pragma unroll
        for (int j = 0; j < 4; ++j) {   // K = 32 codes (32 bytes of a row) per step
          const uint64_t a = smem_desc_sw128(smem + S::kOffA + cc * 16384u + j * 32, 16, 1024);
          const uint64_t w = smem_desc_sw128(smem + S::kOffW + cc * (NT * 128u) + j * 32, 16, 1024);
          mma_f8_ss_warp(tmem, a, w, idesc, (cc | j) ? 1u : 0u);
        }
    } else if (lane == 0) {
      fail_s = 1;
    }
    mma_commit_warp(smem_u32(&acc_full));   // arrives once every MMA issued so far is done
  }
  __syncthreads();
  const bool got = bmm_wait(smem_u32(&acc_full), 0);
  tc_fence_after();
  if ((!got || fail_s) && threadIdx.x == 0) atomicCAS(b.status, 0, MLA_ERR_TIMEOUT);
  const bool ok_all = got && !fail_s;

  // the RoPE part of the decode query (absorption only): the first column tile copies it
  const int n = m0 + r;
  const bool copy_pe = blockIdx.x == 0 && b.pe != nullptr && n < b.N;
  uint4 pe[8];
  if (copy_pe) {
    const uint4* src = reinterpret_cast<const uint4*>(b.pe + static_cast<int64_t>(n) * b.pe_row_stride + h * 64);
#pragma unroll
    for (int j = 0; j < 8; ++j) pe[j] = __ldg(src + j);
    if (b.positions != nullptr) rope_row(pe, __ldg(b.positions + n), b);
  }

  // epilogue: acc * x_scale * w_scale in bf16.  Warp w stages its 32 rows as one 32-row x
  // 64-column tile per 64 output columns (the output map's 128-byte swizzle: row r's 16-byte
  // unit u at r * 128 + ((u ^ (r & 7)) * 16)) in the idle weight / code / x memory, and one
  // lane stores each tile by TMA; rows past N are clipped by the map.
  const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  const int nw0 = m0 + warp * 32;
  static_assert(4 * (NT / 64) * 4096u <= S::kOffX + S::kXStages * 16384u, "the staging tiles fit the idle operands");
  const uint32_t stg = smem + warp * (NT / 64) * 4096u;
  if (ok_all && nw0 < b.N) {
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
        x.x = pack_bf16x2(__uint_as_float(v[0]) * out_scale, __uint_as_float(v[1]) * out_scale);
        x.y = pack_bf16x2(__uint_as_float(v[2]) * out_scale, __uint_as_float(v[3]) * out_scale);
        x.z = pack_bf16x2(__uint_as_float(v[4]) * out_scale, __uint_as_float(v[5]) * out_scale);
        x.w = pack_bf16x2(__uint_as_float(v[6]) * out_scale, __uint_as_float(v[7]) * out_scale);
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
  if (ok_all && copy_pe) {
    uint4* d4 = reinterpret_cast<uint4*>(b.out + static_cast<int64_t>(n) * b.out_row_stride +
                                         static_cast<int64_t>(h) * b.out_head_stride + 512);
#pragma unroll
    for (int j = 0; j < 8; ++j) d4[j] = pe[j];
  }
  if (threadIdx.x == 0) {   // loads still in flight after a failure land before the CTA may exit
    if (issued_w && !got) bmm_wait(smem_u32(&w_full), 0);
    if (!ok)   // each stage's latest load (an older phase of its barrier may alias)
      for (int c = x_issued - S::kXStages < 0 ? 0 : x_issued - S::kXStages; c < x_issued; ++c)
        bmm_wait(smem_u32(&x_full[c % S::kXStages]), (c / S::kXStages) & 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, NT);
  }
}

// absorb: K = 128 -> two 256-column tiles of 512; un-absorb: K = 512 -> one 128-column tile
#define MLA_FP8_ABSORB 128, 256
#define MLA_FP8_UNABSORB 512, 128

// dynamic shared memory of the amax launch when it also computes the schedule
constexpr size_t kAmaxPlanSmem = sizeof(int64_t) * (kAbsorbPlanMaxB + 1) + sizeof(int32_t) * kAbsorbPlanMaxB;

cudaError_t bmm_fp8_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(mla_amax_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kAmaxPlanSmem));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(mla_bmm_fp8_kernel<MLA_FP8_ABSORB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(Fp8BmmShape<MLA_FP8_ABSORB>::kSmem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(mla_bmm_fp8_kernel<MLA_FP8_UNABSORB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(Fp8BmmShape<MLA_FP8_UNABSORB>::kSmem));
}

cudaError_t launch_bmm_fp8(bool absorb, const __nv_bfloat16* x, int64_t x_row_stride, int K, const CUtensorMap& x_map,
                           const CUtensorMap& w_map, const CUtensorMap& o_map, const BmmFp8Params& p, float* partials,
                           cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  {   // the partial maxima of |x| over the N rows of H * K values (and the schedule, if asked)
    const bool plan = p.base.sched_meta != nullptr;
    if (plan && (!absorb || p.base.sched_B < 1 || p.base.sched_B > kAbsorbPlanMaxB || p.base.sched_parts < 1))
      return cudaErrorInvalidValue;
    const size_t smem = plan ? sizeof(int64_t) * (p.base.sched_B + 1) + sizeof(int32_t) * p.base.sched_B : 0;
    const cudaLaunchConfig_t cfg = pdl_config(dim3(kAmaxParts + (plan ? 1 : 0)), dim3(256), smem, stream, attr);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, mla_amax_kernel, x, static_cast<int64_t>(p.base.N),
                                             static_cast<int64_t>(p.base.H) * K / 8, x_row_stride, partials,
                                             p.base);
    if (e != cudaSuccess) return e;
  }
  const unsigned mt = static_cast<unsigned>((p.base.N + 127) / 128);
  if (absorb) {
    const cudaLaunchConfig_t cfg = pdl_config(dim3(512 / 256, p.base.H, mt), dim3(128),
                                              Fp8BmmShape<MLA_FP8_ABSORB>::kSmem, stream, attr);
    return cudaLaunchKernelEx(&cfg, mla_bmm_fp8_kernel<MLA_FP8_ABSORB>, x_map, w_map, o_map, p);
  }
  const cudaLaunchConfig_t cfg = pdl_config(dim3(128 / 128, p.base.H, mt), dim3(128),
                                            Fp8BmmShape<MLA_FP8_UNABSORB>::kSmem, stream, attr);
  return cudaLaunchKernelEx(&cfg, mla_bmm_fp8_kernel<MLA_FP8_UNABSORB>, x_map, w_map, o_map, p);
}

}  // namespace mla
