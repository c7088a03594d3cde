// Absorbed MLA decode on sm_103a: paged latent KV, split-KV segments, tcgen05.
//
// What is computed ("MLA 推理：两条计算路径与 FlashMLA", section "两条等价的路径",
// path 2; "DeepSeekV2之MLA" 4.3): H query heads (times s_q positions) share one
// cached row of 576 values per token; score = <q, kv[0:576]> * scale, softmax
// over the visible tokens, output = sum p_t kv_t[0:512].  Section "decode 注意力变成
// 了计算问题" of the first page fixes the kernel shape: all heads form the M
// dimension of a tensor-core GEMM, each latent tile is read once and used by
// both QK^T and PV on chip, and long contexts are split along the KV axis
// across SMs with the partial results merged by LSE afterwards.
//
// Design on GB300.  A 128-row tile of queries against a 64-token page needs an
// fp32 output accumulator of 128 x 512 -- all 512 TMEM columns of one SM -- so
// the work of one row block is split over a CTA pair in one cluster:
//   * the S-CTA (even cluster rank) keeps Q in TMEM (288 columns, A operand),
//     computes S = Q K^T for each page with tcgen05 (A from TMEM, B = the page in
//     shared memory), runs the online softmax in fp32, and ships P (bf16, in the
//     MMA operand layout) plus the per-row rescale factors to its partner with a
//     shared-to-shared bulk copy;
//   * the O-CTA (odd rank) keeps O (128 x 512 fp32) in TMEM, loads the value
//     part of each page, runs O += P V with tcgen05, rescales O only when a row
//     maximum grew by more than 2^8 (exact: the final normalisation uses the same
//     reference maximum), and writes the normalised output (bf16) or, for a
//     split request, an fp32 partial that the combine kernel merges.
// Rows beyond 128 (s_q * H > 128) go to further pairs of the same cluster, which
// walk the same pages at the same time so that a page is fetched from HBM once.
// A cluster is one "part" of the split schedule and walks the segments the
// metadata assigns to it.
//
// Roles inside a CTA (256 threads): warp 0 = TMA producer, warp 1 = MMA issuer,
// warp 2 = credit forwarder (O-CTA), warps 4..7 = softmax (S-CTA) or
// rescale/epilogue (O-CTA) warpgroup, one query row per thread.
// Every barrier wait is bounded; on expiry the CTA records MLA_ERR_TIMEOUT,
// raises an abort flag in every CTA of its cluster, drains what it has in
// flight and exits.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "mla_kernels.h"
#include "mla_ptx.cuh"

namespace mla {

namespace {

constexpr int kThreads = 256;
constexpr uint32_t kKStageBytes = 9 * 8192;          // 64 tokens x 576 dims, 9 swizzled chunks
constexpr uint32_t kVStageBytes = 8 * 8192;          // 64 tokens x 512 dims
constexpr uint32_t kPBytes = 128 * 128;              // P: 128 rows x 64 tokens bf16
constexpr uint32_t kPktAlpha = kPBytes;              // float[128]
constexpr uint32_t kPktInvL = kPBytes + 512;         // float[128]
constexpr uint32_t kPktFlags = kPBytes + 1024;       // uint32[4]
constexpr uint32_t kPktBytes = kPBytes + 1024 + 16;  // bytes moved per page
constexpr uint32_t kPktStride = 18 * 1024;
// dynamic shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t kOffStage = 0;                    // 2 K stages (S-CTA) or 2 V stages (O-CTA)
constexpr uint32_t kOffRecv = 2 * kVStageBytes;      // O-CTA: 2 packet receive slots
constexpr uint32_t kOffSend = 2 * kKStageBytes;      // S-CTA: 2 packet staging slots
constexpr uint32_t kSmemBytes = kOffSend + 2 * kPktStride;
constexpr uint32_t kQCol = 0, kSCol0 = 320;          // S-CTA TMEM columns: Q [0,288), S buffers 320, 384
constexpr float kRescaleLog2 = 8.0f;                 // rebase the row max when it grows by more than 2^8
constexpr int kPrefetchAhead = 4;                    // pages prefetched into L2 ahead of the loads
constexpr uint64_t kTimeoutNs = 500ull * 1000 * 1000;
constexpr float kLn2 = 0.69314718055994530942f;

static_assert(kOffRecv + 2 * kPktStride <= kSmemBytes, "O-CTA layout");
static_assert(kPktBytes % 16 == 0 && kPktStride % 1024 == 0, "packet alignment");

struct Bars {
  uint64_t full[2];       // page landed (S: K, O: V)
  uint64_t empty[2];      // stage free again
  uint64_t s_full[2];     // S-CTA: S = QK^T ready in TMEM
  uint64_t s_empty[2];    // S-CTA: S read by the softmax warps
  uint64_t q_full;        // S-CTA: Q of the segment stored in TMEM
  uint64_t credit[2];     // S-CTA: the partner's receive slot is free (remote arrivals)
  uint64_t p_full[2];     // O-CTA: packet received (bulk-copy bytes)
  uint64_t p_free[2];     // O-CTA: PV MMAs that read a packet slot are done
  uint64_t o_full;        // O-CTA: the segment's last PV MMAs are done
  uint64_t o_free;        // O-CTA: epilogue finished reading O
  uint64_t o_sync;        // O-CTA: all PV MMAs issued so far are done (before a rescale)
  uint64_t corr_go;       // O-CTA: command for the rescale/epilogue warpgroup
  uint64_t corr_done;     // O-CTA: rescale finished
  uint64_t drain;         // both: final MMA completion
};

struct __align__(16) Shared {
  Bars bar;
  uint32_t tmem_base;
  volatile int abort;
  int cmd;                // O-CTA command: 1 = rescale (slot in cmd_arg), 2 = epilogue, 3 = exit
  int cmd_arg;
  __align__(16) float inv_l[128];   // O-CTA: 1/l of the segment's rows (16-byte vector copies)
};
static_assert(offsetof(Shared, inv_l) % 16 == 0, "inv_l is copied with 16-byte shared stores");

struct Segment {
  int b, kb, ke, split;   // request, page range, split index within the request
};

// Walks the segments of one part in order (same walk in every role).
struct SegmentWalker {
  const DecodeParams* p;
  int b_last, k_end, b, kb, split0;
  bool first, done;
  __device__ void init(const DecodeParams& prm, int part) {
    p = &prm;
    const int* m = prm.meta + part * 8;
    b = m[0];
    kb = m[1];
    b_last = m[2];
    k_end = m[3];
    split0 = m[4];
    first = true;
    done = (b < 0);
  }
  __device__ static int pages_of(int L) { return L > 0 ? (L + 63) / 64 : 0; }
  __device__ bool next(Segment& s) {
    while (!done) {
      if (b > b_last) { done = true; break; }
      const int nb = pages_of(__ldg(p->seqlens + b));
      const int k0 = first ? kb : 0;
      const int k1 = (b == b_last) ? k_end : nb;
      const int sp = first ? split0 : 0;
      first = false;
      const int cur = b;
      ++b;
      if (k1 > k0) {
        s.b = cur; s.kb = k0; s.ke = k1; s.split = sp;
        return true;
      }
    }
    return false;
  }
};

__device__ __forceinline__ void raise_abort(Shared& sh, int* status, int code, uint32_t cluster_ctas) {
  if (!sh.abort) {
    atomicCAS(status, 0, code);
    for (uint32_t r = 0; r < cluster_ctas; ++r)
      st_cluster_u32(map_to_rank(smem_u32(const_cast<int*>(&sh.abort)), r), 1u);
  }
  sh.abort = 1;
}

// Bounded wait.  Returns false on abort or timeout (after raising the abort).
__device__ __noinline__ bool wait_bar(Shared& sh, uint32_t bar, uint32_t parity, int* status,
                                      uint32_t cluster_ctas, bool cluster_scope = false) {
  if (cluster_scope ? mbar_test_cluster(bar, parity) : mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (cluster_scope ? mbar_test_cluster(bar, parity) : mbar_test(bar, parity)) return true;
    if (sh.abort) return false;
    if (global_timer_ns() - t0 > kTimeoutNs) {
      raise_abort(sh, status, MLA_ERR_TIMEOUT, cluster_ctas);
      return false;
    }
  }
}
// All 32 lanes wait; the result is made uniform across the warp.
__device__ __forceinline__ bool warp_wait(Shared& sh, uint32_t bar, uint32_t parity, int* status, uint32_t cluster_ctas,
                                          bool cluster_scope = false) {
  const bool ok = wait_bar(sh, bar, parity, status, cluster_ctas, cluster_scope);
  return __all_sync(0xffffffffu, ok);
}
// Bounded wait that ignores the abort flag: used to drain operations in flight.
__device__ __noinline__ void drain_bar(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > kTimeoutNs) return;
  }
}

// Page id of page k of request b, or -1 (and a recorded bounds error) if the
// table entry is outside [0, num_blocks) or k is past the table's width.
__device__ __forceinline__ int request_block(const DecodeParams& p, int b, int k) {
  if (k >= p.max_blocks) {
    atomicCAS(p.status, 0, MLA_ERR_DEVICE_BOUNDS);
    return -1;
  }
  int blk = __ldg(p.block_table + static_cast<int64_t>(b) * p.max_blocks + k);
  if (blk < 0 || blk >= p.num_blocks) {
    atomicCAS(p.status, 0, MLA_ERR_DEVICE_BOUNDS);
    blk = -1;   // the TMA then reads out-of-range rows, which it fills with zeros
  }
  return blk;
}

// ------------------------------------------------------------------ S-CTA --
__device__ void s_cta_producer(const DecodeParams& p, const CUtensorMap* kv_map, Shared& sh, uint32_t smem,
                               int part, uint32_t cl, bool prefetcher) {
  SegmentWalker w;
  w.init(p, part);
  Segment s;
  uint32_t T = 0;
  uint32_t issued_mask_phase[2] = {0, 0};
  int issued[2] = {0, 0};
  const uint64_t policy = l2_policy_evict_first();
  bool ok = true;
  while (ok && w.next(s)) {
    if (prefetcher) {
      for (int k = s.kb; k < s.ke && k < s.kb + kPrefetchAhead && k < p.max_blocks; ++k) {
        const int blk = __ldg(p.block_table + static_cast<int64_t>(s.b) * p.max_blocks + k);
        if (blk >= 0 && blk < p.num_blocks) prefetch_l2(p.kv + static_cast<int64_t>(blk) * 64 * 576, kKStageBytes);
      }
    }
    for (int k = s.kb; k < s.ke; ++k, ++T) {
      const uint32_t st = T & 1, ph = (T >> 1) & 1;
      if (!wait_bar(sh, smem_u32(&sh.bar.empty[st]), ph ^ 1, p.status, cl)) { ok = false; break; }
      if (prefetcher && k + kPrefetchAhead < s.ke && k + kPrefetchAhead < p.max_blocks) {
        const int blk = __ldg(p.block_table + static_cast<int64_t>(s.b) * p.max_blocks + k + kPrefetchAhead);
        if (blk >= 0 && blk < p.num_blocks) prefetch_l2(p.kv + static_cast<int64_t>(blk) * 64 * 576, kKStageBytes);
      }
      if (p.withhold_first_load && T == 0) continue;   // test hook: this page never arrives
      const int blk = request_block(p, s.b, k);
      const uint32_t full = smem_u32(&sh.bar.full[st]);
      mbar_arrive_expect_tx(full, kKStageBytes);
      const uint32_t dst = smem + kOffStage + st * kKStageBytes;
      for (int c = 0; c < 9; ++c) tma_load_2d_hint(dst + c * 8192, kv_map, full, c * 64, blk * 64, policy);
      issued[st] = 1;
      issued_mask_phase[st] = ph;
    }
  }
  // drain: loads still in flight land before the CTA may exit
  for (int st = 0; st < 2; ++st)
    if (issued[st]) drain_bar(smem_u32(&sh.bar.full[st]), issued_mask_phase[st]);
}

// Warp 1 of the S-CTA; all 32 lanes run the loop, one elected lane issues.
__device__ void s_cta_mma(const DecodeParams& p, Shared& sh, uint32_t smem, int part, uint32_t cl) {
  SegmentWalker w;
  w.init(p, part);
  Segment s;
  uint32_t T = 0, seg = 0;
  const uint32_t tmem = sh.tmem_base;
  constexpr uint32_t idesc = idesc_bf16_f32(128, 64, 0, 0);
  bool ok = true, any = false;
  while (ok && w.next(s)) {
    if (!warp_wait(sh, smem_u32(&sh.bar.q_full), seg & 1, p.status, cl)) break;
    for (int k = s.kb; k < s.ke; ++k, ++T) {
      const uint32_t st = T & 1, ph = (T >> 1) & 1;
      if (!warp_wait(sh, smem_u32(&sh.bar.full[st]), ph, p.status, cl)) { ok = false; break; }
      if (!warp_wait(sh, smem_u32(&sh.bar.s_empty[st]), ph ^ 1, p.status, cl)) { ok = false; break; }
      tc_fence_after();
      const uint32_t kstage = smem + kOffStage + st * kKStageBytes;
      const uint32_t d = tmem + kSCol0 + st * 64;
#pragma unroll
      for (int kk = 0; kk < 36; ++kk) {
        const uint64_t bdesc = smem_desc_sw128(kstage + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024);
        mma_bf16_ts_warp(d, tmem + kQCol + kk * 8, bdesc, idesc, kk > 0 ? 1u : 0u);
      }
      mma_commit_warp(smem_u32(&sh.bar.empty[st]));
      mma_commit_warp(smem_u32(&sh.bar.s_full[st]));
      any = true;
    }
    ++seg;
  }
  if (any) {
    mma_commit_warp(smem_u32(&sh.bar.drain));
    drain_bar(smem_u32(&sh.bar.drain), 0);
  }
  __syncwarp();
}

__device__ void s_cta_softmax(const DecodeParams& p, Shared& sh, uint32_t smem, int part, uint32_t cl, int rb,
                              uint32_t peer) {
  const int r = threadIdx.x - 128;          // row within the block == TMEM lane
  const int wq = r >> 5, lane = r & 31;
  const int g = rb * 128 + r;               // row within the request: i * H + h
  const bool row_valid = g < p.rows;
  const int pos_i = row_valid ? g / p.H : 0;
  const uint32_t tmem_lane = sh.tmem_base + (static_cast<uint32_t>(wq * 32) << 16);
  const uint32_t peer_recv = map_to_rank(smem + kOffRecv, peer);
  const uint32_t peer_pfull0 = map_to_rank(smem_u32(&sh.bar.p_full[0]), peer);
  const uint32_t peer_pfull1 = map_to_rank(smem_u32(&sh.bar.p_full[1]), peer);
  SegmentWalker w;
  w.init(p, part);
  Segment s;
  uint32_t T = 0;
  bool ok = true;
  while (ok && w.next(s)) {
    const int L = __ldg(p.seqlens + s.b);
    int vis = L;
    if (p.causal && row_valid) vis = L - p.s_q + pos_i + 1;
    // Q of this request into TMEM columns [0, 288): one row per thread.
    {
      const int gq = row_valid ? g : 0;
      const uint4* src = reinterpret_cast<const uint4*>(p.q + (static_cast<int64_t>(s.b) * p.rows + gq) * 576);
#pragma unroll 1
      for (int c = 0; c < 9; ++c) {
        uint32_t v[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint4 x = row_valid ? __ldg(src + c * 8 + j) : make_uint4(0, 0, 0, 0);
          v[4 * j] = x.x; v[4 * j + 1] = x.y; v[4 * j + 2] = x.z; v[4 * j + 3] = x.w;
        }
        tmem_st32(tmem_lane + kQCol + c * 32, v);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.bar.q_full));
    }
    float m_ref = -INFINITY, l = 0.f;
    for (int k = s.kb; k < s.ke; ++k, ++T) {
      const uint32_t sb = T & 1, ph = (T >> 1) & 1;
      const bool got = wait_bar(sh, smem_u32(&sh.bar.s_full[sb]), ph, p.status, cl);
      if (named_bar_or(1, 128, !got)) { ok = false; break; }   // same decision in all 128 threads
      tc_fence_after();
      uint32_t sr[64];
      tmem_ld32(tmem_lane + kSCol0 + sb * 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(tmem_lane + kSCol0 + sb * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.bar.s_empty[sb]));

      // scaled, masked scores (log2 units); slots at or past `vis` become -inf
      const int t0 = k * 64;
      const int nvalid = vis - t0;              // columns c < nvalid are visible
      float x[64];
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        x[c] = (c < nvalid) ? __uint_as_float(sr[c]) * p.scale_log2 : -INFINITY;
        mt = fmaxf(mt, x[c]);
      }
      const float m_new = fmaxf(m_ref, mt);
      float alpha = 1.f;
      const bool rebase = m_new > m_ref + kRescaleLog2;
      if (rebase) {
        alpha = fast_exp2(m_ref - m_new);       // 0 when m_ref = -inf
        m_ref = m_new;
      }
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      uint32_t pk[32];
      float psum = 0.f;
#pragma unroll
      for (int c = 0; c < 32; ++c) {   // l sums the fp32 probabilities; P goes to the MMA in bf16
        const float e0 = fast_exp2(x[2 * c] - m_use), e1 = fast_exp2(x[2 * c + 1] - m_use);
        pk[c] = pack_bf16x2(e0, e1);
        psum += e0 + e1;
      }
      l = l * alpha + psum;
      const bool last = (k == s.ke - 1);
      const bool first = (k == s.kb);
      const uint32_t need = __ballot_sync(0xffffffffu, rebase && !first);

      // packet into the staging slot, then one bulk copy to the partner
      const uint32_t slot = smem + kOffSend + sb * kPktStride;
      if (r == 0) bulk_wait_group_read<1>();     // the copy that used this slot two pages ago has read it
      named_bar_sync(1, 128);
      {
        const uint32_t row = slot + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t a = row + ((c ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                       :: "r"(a), "r"(pk[4 * c]), "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3]) : "memory");
        }
        asm volatile("st.shared.f32 [%0], %1;" :: "r"(slot + kPktAlpha + r * 4), "f"(alpha) : "memory");
        if (last) {
          const float inv_l = l > 0.f ? 1.f / l : 0.f;
          asm volatile("st.shared.f32 [%0], %1;" :: "r"(slot + kPktInvL + r * 4), "f"(inv_l) : "memory");
        }
        if (lane == 0) asm volatile("st.shared.u32 [%0], %1;" :: "r"(slot + kPktFlags + wq * 4), "r"(need) : "memory");
      }
      fence_proxy_async_smem();
      bool credit_ok = true;
      if (r == 0) credit_ok = wait_bar(sh, smem_u32(&sh.bar.credit[sb]), ph ^ 1, p.status, cl, true);
      if (named_bar_or(1, 128, !credit_ok)) { ok = false; break; }
      if (r == 0) {
        bulk_copy_to_cluster(peer_recv + sb * kPktStride, slot, kPktBytes, sb ? peer_pfull1 : peer_pfull0);
        bulk_commit_group();
      }
    }
    if (!ok) break;
    if (row_valid) {
      const float lse = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
      const int ns0 = __ldg(p.num_splits + s.b);
      const int nsplit = __ldg(p.num_splits + s.b + 1) - ns0;
      if (nsplit == 1)
        p.lse[static_cast<int64_t>(s.b) * p.rows + g] = lse;
      else
        p.lse_part[static_cast<int64_t>(ns0 + s.split) * p.rows + g] = lse;
    }
  }
  if (r == 0) bulk_wait_group<0>();
}

// ------------------------------------------------------------------ O-CTA --
__device__ void o_cta_producer(const DecodeParams& p, const CUtensorMap* kv_map, Shared& sh, uint32_t smem,
                               int part, uint32_t cl) {
  SegmentWalker w;
  w.init(p, part);
  Segment s;
  uint32_t T = 0;
  int issued[2] = {0, 0};
  uint32_t issued_phase[2] = {0, 0};
  const uint64_t policy = l2_policy_evict_first();
  bool ok = true;
  while (ok && w.next(s)) {
    for (int k = s.kb; k < s.ke; ++k, ++T) {
      const uint32_t st = T & 1, ph = (T >> 1) & 1;
      if (!wait_bar(sh, smem_u32(&sh.bar.empty[st]), ph ^ 1, p.status, cl)) { ok = false; break; }
      const int blk = request_block(p, s.b, k);
      const uint32_t full = smem_u32(&sh.bar.full[st]);
      mbar_arrive_expect_tx(full, kVStageBytes);
      const uint32_t dst = smem + kOffStage + st * kVStageBytes;
      for (int c = 0; c < 8; ++c) tma_load_2d_hint(dst + c * 8192, kv_map, full, c * 64, blk * 64, policy);
      issued[st] = 1;
      issued_phase[st] = ph;
    }
  }
  for (int st = 0; st < 2; ++st)
    if (issued[st]) drain_bar(smem_u32(&sh.bar.full[st]), issued_phase[st]);
}

// Warp 1 of the O-CTA (all 32 lanes enter; lane 0 issues).
__device__ void o_cta_mma(const DecodeParams& p, Shared& sh, uint32_t smem, int part, uint32_t cl) {
  const int lane = threadIdx.x & 31;
  SegmentWalker w;
  w.init(p, part);
  Segment s;
  uint32_t T = 0, seg = 0, ncmd = 0, nresc = 0;
  const uint32_t tmem = sh.tmem_base;
  constexpr uint32_t idesc = idesc_bf16_f32(128, 256, 0, 1);
  bool ok = true, any = false;
  while (ok && w.next(s)) {
    if (seg > 0 && !warp_wait(sh, smem_u32(&sh.bar.o_free), (seg - 1) & 1, p.status, cl)) break;
    const int L = __ldg(p.seqlens + s.b);
    for (int k = s.kb; k < s.ke; ++k, ++T) {
      const uint32_t st = T & 1, ph = (T >> 1) & 1;
      const uint32_t vstage = smem + kOffStage + st * kVStageBytes;
      const uint32_t pkt = smem + kOffRecv + st * kPktStride;
      if (lane == 0) mbar_arrive_expect_tx(smem_u32(&sh.bar.p_full[st]), kPktBytes);
      __syncwarp();
      if (!warp_wait(sh, smem_u32(&sh.bar.full[st]), ph, p.status, cl)) { ok = false; break; }
      if (!warp_wait(sh, smem_u32(&sh.bar.p_full[st]), ph, p.status, cl, true)) { ok = false; break; }
      // tail page: zero the value rows past the sequence end up to the next 16-row
      // boundary, so that P = 0 never meets a non-finite value in the MMA
      const int nvalid = min(64, L - k * 64);
      const int krows = (nvalid + 15) & ~15;
      if (nvalid < krows) {
        const int nz = krows - nvalid;                 // rows to clear, < 16
        for (int i = lane; i < nz * 8 * 8; i += 32) {  // rows x chunks x 16-byte units
          const int row = nvalid + i / 64, chunk = (i / 8) % 8, u = i % 8;
          asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};"
                       :: "r"(vstage + chunk * 8192 + row * 128 + u * 16), "r"(0u) : "memory");
        }
        fence_proxy_async_smem();
      }
      const bool last = (k == s.ke - 1);
      if (last)     // keep 1/l of the segment's rows before the slot can be reused
        st_shared_v4(smem_u32(&sh.inv_l[lane * 4]), ld_shared_v4(pkt + kPktInvL + lane * 16));
      __syncwarp();
      uint32_t need = 0;
      if (k != s.kb) {
        const uint4 f = ld_shared_v4(pkt + kPktFlags);
        need = f.x | f.y | f.z | f.w;
      }
      if (need) {   // a row maximum was rebased: scale O by alpha before adding this page
        mma_commit_warp(smem_u32(&sh.bar.o_sync));
        if (!warp_wait(sh, smem_u32(&sh.bar.o_sync), nresc & 1, p.status, cl)) { ok = false; break; }
        if (lane == 0) {
          sh.cmd = 1;
          sh.cmd_arg = static_cast<int>(st);
          mbar_arrive(smem_u32(&sh.bar.corr_go));
        }
        ++ncmd;
        __syncwarp();
        if (!warp_wait(sh, smem_u32(&sh.bar.corr_done), nresc & 1, p.status, cl)) { ok = false; break; }
        ++nresc;
      }
      tc_fence_after();
      {
        const int ksteps = krows / 16;
        for (int js = 0; js < ksteps; ++js) {
          const uint64_t adesc = smem_desc_sw128(pkt + js * 32, 16, 1024);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const uint64_t bdesc = smem_desc_sw128(vstage + h2 * 4 * 8192 + js * 2048, 8192, 1024);
            mma_bf16_ss_warp(tmem + h2 * 256, adesc, bdesc, idesc, (k == s.kb && js == 0) ? 0u : 1u);
          }
        }
        mma_commit_warp(smem_u32(&sh.bar.empty[st]));
        mma_commit_warp(smem_u32(&sh.bar.p_free[st]));
        if (last) mma_commit_warp(smem_u32(&sh.bar.o_full));
      }
      any = true;
      __syncwarp();
      if (last) {
        if (lane == 0) {
          sh.cmd = 2;
          sh.cmd_arg = static_cast<int>(seg);
          mbar_arrive(smem_u32(&sh.bar.corr_go));
        }
        ++ncmd;
      }
    }
    ++seg;
  }
  // wait for the epilogue of the last segment before posting the exit command
  if (ok && seg > 0) warp_wait(sh, smem_u32(&sh.bar.o_free), (seg - 1) & 1, p.status, cl);
  if (any) {
    mma_commit_warp(smem_u32(&sh.bar.drain));
    drain_bar(smem_u32(&sh.bar.drain), 0);
  }
  __syncwarp();
  if (lane == 0) {
    sh.cmd = 3;
    mbar_arrive(smem_u32(&sh.bar.corr_go));
  }
  __syncwarp();
  (void)ncmd;
}

// Warp 2 of the O-CTA: returns each packet slot to the S-CTA once the MMAs reading it are done.
__device__ void o_cta_forwarder(const DecodeParams& p, Shared& sh, int part, uint32_t cl, uint32_t peer) {
  SegmentWalker w;
  w.init(p, part);
  Segment s;
  uint32_t T = 0;
  const uint32_t credit0 = map_to_rank(smem_u32(&sh.bar.credit[0]), peer);
  const uint32_t credit1 = map_to_rank(smem_u32(&sh.bar.credit[1]), peer);
  bool ok = true;
  while (ok && w.next(s)) {
    for (int k = s.kb; k < s.ke; ++k, ++T) {
      const uint32_t st = T & 1, ph = (T >> 1) & 1;
      if (!wait_bar(sh, smem_u32(&sh.bar.p_free[st]), ph, p.status, cl)) { ok = false; break; }
      mbar_arrive_remote(st ? credit1 : credit0);
    }
  }
}

// Warps 4..7 of the O-CTA: rescale O rows, or normalise and store a finished segment.
__device__ void o_cta_epilogue(const DecodeParams& p, Shared& sh, uint32_t smem, int part, uint32_t cl, int rb) {
  const int r = threadIdx.x - 128;
  const int wq = r >> 5, lane = r & 31;
  const int g = rb * 128 + r;
  const bool row_valid = g < p.rows;
  const uint32_t tmem_lane = sh.tmem_base + (static_cast<uint32_t>(wq * 32) << 16);
  SegmentWalker w;
  w.init(p, part);
  Segment s;
  uint32_t ncmd = 0, seg = 0;
  bool have_seg = w.next(s);
  while (true) {
    if (!warp_wait(sh, smem_u32(&sh.bar.corr_go), ncmd & 1, p.status, cl)) break;
    ++ncmd;
    const int cmd = sh.cmd, arg = sh.cmd_arg;
    if (cmd == 3) break;
    if (cmd == 1) {
      const uint32_t pkt = smem + kOffRecv + arg * kPktStride;
      const float alpha = ld_shared_f32(pkt + kPktAlpha + r * 4);
      tc_fence_after();
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < 512; c += 32) {
          uint32_t v[32];
          tmem_ld32(tmem_lane + c, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
          tmem_st32(tmem_lane + c, v);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.bar.corr_done));
      continue;
    }
    // cmd == 2: epilogue of segment `seg`
    if (!have_seg) break;
    if (!warp_wait(sh, smem_u32(&sh.bar.o_full), seg & 1, p.status, cl)) break;
    tc_fence_after();
    const float inv_l = sh.inv_l[r];
    const int ns0 = __ldg(p.num_splits + s.b);
    const int nsplit = __ldg(p.num_splits + s.b + 1) - ns0;
    const bool final_out = (nsplit == 1);
    __nv_bfloat16* orow = p.out + (static_cast<int64_t>(s.b) * p.rows + g) * 512;
    float* prow = p.o_part + (static_cast<int64_t>(ns0 + s.split) * p.rows + g) * 512;
#pragma unroll 1
    for (int c = 0; c < 512; c += 32) {
      uint32_t v[32];
      tmem_ld32(tmem_lane + c, v);
      tmem_wait_ld();
      if (c == 480) {   // everything read: O may be overwritten by the next segment
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.bar.o_free));
      }
      if (!row_valid) continue;
      if (final_out) {
        uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint4 u;
          u.x = pack_bf16x2(__uint_as_float(v[8 * j + 0]) * inv_l, __uint_as_float(v[8 * j + 1]) * inv_l);
          u.y = pack_bf16x2(__uint_as_float(v[8 * j + 2]) * inv_l, __uint_as_float(v[8 * j + 3]) * inv_l);
          u.z = pack_bf16x2(__uint_as_float(v[8 * j + 4]) * inv_l, __uint_as_float(v[8 * j + 5]) * inv_l);
          u.w = pack_bf16x2(__uint_as_float(v[8 * j + 6]) * inv_l, __uint_as_float(v[8 * j + 7]) * inv_l);
          dst[j] = u;
        }
      } else {
        float4* dst = reinterpret_cast<float4*>(prow + c);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          dst[j] = make_float4(__uint_as_float(v[4 * j]) * inv_l, __uint_as_float(v[4 * j + 1]) * inv_l,
                               __uint_as_float(v[4 * j + 2]) * inv_l, __uint_as_float(v[4 * j + 3]) * inv_l);
      }
    }
    ++seg;
    have_seg = w.next(s);
  }
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
mla_decode_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t dyn_smem[];
  __shared__ Shared sh;
  const uint32_t smem = (smem_u32(dyn_smem) + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5;
  const uint32_t rank = cluster_ctarank();
  const uint32_t cl = 2u * static_cast<uint32_t>(p.n_rb);   // CTAs per cluster
  const int part = static_cast<int>(blockIdx.x / cl);
  const int rb = static_cast<int>(rank >> 1);
  const bool is_s = (rank & 1u) == 0;
  const uint32_t peer = rank ^ 1u;

  if (threadIdx.x == 0) {
    sh.abort = 0;
    sh.cmd = 0;
    mbar_init(smem_u32(&sh.bar.full[0]), 1);
    mbar_init(smem_u32(&sh.bar.full[1]), 1);
    mbar_init(smem_u32(&sh.bar.empty[0]), 1);
    mbar_init(smem_u32(&sh.bar.empty[1]), 1);
    mbar_init(smem_u32(&sh.bar.s_full[0]), 1);
    mbar_init(smem_u32(&sh.bar.s_full[1]), 1);
    mbar_init(smem_u32(&sh.bar.s_empty[0]), 4);
    mbar_init(smem_u32(&sh.bar.s_empty[1]), 4);
    mbar_init(smem_u32(&sh.bar.q_full), 4);
    mbar_init(smem_u32(&sh.bar.credit[0]), 1);
    mbar_init(smem_u32(&sh.bar.credit[1]), 1);
    mbar_init(smem_u32(&sh.bar.p_full[0]), 1);
    mbar_init(smem_u32(&sh.bar.p_full[1]), 1);
    mbar_init(smem_u32(&sh.bar.p_free[0]), 1);
    mbar_init(smem_u32(&sh.bar.p_free[1]), 1);
    mbar_init(smem_u32(&sh.bar.o_full), 1);
    mbar_init(smem_u32(&sh.bar.o_free), 4);
    mbar_init(smem_u32(&sh.bar.o_sync), 1);
    mbar_init(smem_u32(&sh.bar.corr_go), 1);
    mbar_init(smem_u32(&sh.bar.corr_done), 4);
    mbar_init(smem_u32(&sh.bar.drain), 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (warp == 0) tmem_alloc(smem_u32(&sh.tmem_base), 512);
  tc_fence_before();
  __syncthreads();
  cluster_sync();        // every barrier of the cluster is initialised before any remote use
  tc_fence_after();

  if (is_s) {
    if (warp == 0) {
      if ((threadIdx.x & 31) == 0) s_cta_producer(p, &kv_map, sh, smem, part, cl, rb == 0);
    } else if (warp == 1) {
      s_cta_mma(p, sh, smem, part, cl);
    } else if (warp >= 4) {
      s_cta_softmax(p, sh, smem, part, cl, rb, peer);
    }
  } else {
    if (warp == 0) {
      if ((threadIdx.x & 31) == 0) o_cta_producer(p, &kv_map, sh, smem, part, cl);
    } else if (warp == 1) {
      o_cta_mma(p, sh, smem, part, cl);
    } else if (warp == 2) {
      if ((threadIdx.x & 31) == 0) o_cta_forwarder(p, sh, part, cl, peer);
    } else if (warp >= 4) {
      o_cta_epilogue(p, sh, smem, part, cl, rb);
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();        // no CTA leaves while a partner may still touch its shared memory
  __syncwarp();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(sh.tmem_base, 512);
  }
}

cudaError_t decode_set_attributes() {
  return cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kSmemBytes + 1024));
}

static cudaLaunchConfig_t decode_config(int grid_ctas, int cluster_ctas, cudaStream_t stream,
                                        cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster_ctas);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(grid_ctas), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes + 1024;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

int decode_max_clusters(int cluster_ctas) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = decode_config(cluster_ctas, cluster_ctas, nullptr, attr);
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, mla_decode_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return clusters;
}

cudaError_t launch_decode(const CUtensorMap& kv_map, const DecodeParams& p, int cluster_ctas, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = decode_config(p.num_parts * cluster_ctas, cluster_ctas, stream, attr);
  return cudaLaunchKernelEx(&cfg, mla_decode_kernel, kv_map, p);
}

}  // namespace mla
