// RoPE of the decode query's q_pe part, shared by the bf16 and the FP8 absorption kernels.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "mla_kernels.h"
#include "mla_ptx.cuh"

namespace mla {

// RoPE of one q_pe row in place (64 bf16 values as 32 interleaved pairs; the page's tiny
// example and "DeepSeekV2之MLA" 4.2: the pair (x[2j], x[2j+1]) turns by the angle
// pos * theta^(-2j/64)).  The angle is carried as a float pair: pos is exact in fp32, the
// product with the inverse frequency (itself a float pair) keeps its rounding error via
// fma, and the reduction by 2*pi subtracts k * 2*pi in two parts (Cody and Waite's
// method), so that the argument of the sine and cosine stays within ~1e-7 rad of the
// exact angle for positions up to 2^24.
__device__ __forceinline__ void rope_row(uint4 (&pe)[8], int pos, const BmmParams& p) {
  const float fp = static_cast<float>(pos);
  const float inv_two_pi = 1.0f / p.two_pi_hi;
  uint32_t* w = reinterpret_cast<uint32_t*>(pe);
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float a_hi = fp * p.rope_hi[j];
    const float a_lo = fmaf(fp, p.rope_lo[j], fmaf(fp, p.rope_hi[j], -a_hi));
    const float k = rintf(a_hi * inv_two_pi);
    const float r = fmaf(-k, p.two_pi_lo, fmaf(-k, p.two_pi_hi, a_hi)) + a_lo;
    float sn, cs;
    __sincosf(r, &sn, &cs);   // |r| <= pi + 1e-6: the hardware sine/cosine, absolute error < 2^-21
    const float x0 = bf16_lo(w[j]), x1 = bf16_hi(w[j]);
    w[j] = pack_bf16x2(fmaf(x0, cs, -x1 * sn), fmaf(x0, sn, x1 * cs));
  }
}

}  // namespace mla
