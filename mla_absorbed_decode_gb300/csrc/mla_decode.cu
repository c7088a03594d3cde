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
//   * the S-CTA (even cluster rank) keeps Q in TMEM (288 columns, the MMA's A
//     operand; a segment's q rows arrive by TMA through the same two stages as the
//     pages, 64 rows per stage, and the softmax warps copy them into TMEM),
//     computes S = Q K^T for each page with tcgen05 (B = the page in
//     shared memory, two pages in flight), and runs the online softmax in fp32
//     with two warpgroups that split the page's 64 columns.  It stages P (bf16,
//     already in the MMA operand layout) and the per-row rescale factors in its
//     shared memory and ships them to its partner with one shared-to-shared bulk
//     copy per page (many small remote stores are several times slower);
//   * the O-CTA (odd rank) keeps O (128 x 512 fp32) in TMEM, loads the value
//     part of each page (two in flight), runs O += P V with tcgen05, rescales O
//     only when a row maximum grew by more than 2^8 (exact: the final
//     normalisation uses the same reference maximum), and writes the normalised
//     output (bf16) or, for a split request, an fp32 partial that the combine
//     kernel merges.
// Both CTAs load a page stage in two parts and release each part as soon as the
// MMAs that read it are done (S-CTA: chunks 0..4 and 5..8 of the 576 dims; O-CTA:
// value chunks 0..3 and 4..7), so the refill of the first part overlaps the MMAs
// on the second.
// Rows beyond 128 (s_q * H > 128) go to further pairs of the same cluster, which
// walk the same pages at the same time so that a page is fetched from HBM once.
// A cluster is one "part" of the split schedule and walks the segments the
// metadata assigns to it.
//
// Roles (384 threads): warp 0 = TMA producer, warp 1 = MMA issuer (warp-uniform,
// one elected lane issues), warp 2 = credit forwarder (O-CTA), warps 4..7 and
// 8..11 = two softmax (S-CTA) or rescale/epilogue (O-CTA) warpgroups; a thread
// of a warpgroup owns one query row (its TMEM lane).  The sparse decode runs 512 threads:
// two lookup warps per CTA find its pages' cache rows (row_lookup) and four gathering warps
// load them by TMA (tile::gather4, s_producer_gather / o_producer_gather).
// Every barrier wait is bounded; on expiry the CTA records MLA_ERR_TIMEOUT,
// raises an abort flag in every CTA of its cluster, drains what it has in
// flight and exits.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <climits>
#include <stddef.h>
#include <stdint.h>

#include "mla_kernels.h"
#include "mla_ptx.cuh"

namespace mla {

namespace {

constexpr int kThreads = 384;          // 12 warps; the sparse decode runs 16 (see gather_slot, lookup_half)
template <bool kSparse, bool kF8>
constexpr int threads_of() { return kSparse ? 512 : kThreads; }
constexpr int kMaxStages = 4;                         // barrier slots: the deepest page ring
constexpr int kSlots = 4;                             // O-CTA packet receive slots: a slot's credit
                                                      // round trip over DSMEM is hidden 4 pages deep
constexpr int kRowSlots = 4;                          // sparse: pages of looked-up cache rows in flight
constexpr uint32_t kChunk = 8192;                     // one swizzled chunk of a page: 64 rows x 128 B
constexpr uint32_t kPBytes = 128 * 128;               // P: 128 rows x 128 B in the MMA A layout (bf16: 64
                                                      // tokens; FP8: hi and lo codes of 64 tokens)
constexpr uint32_t kPktAlpha = kPBytes;               // float[128] rescale factor per row
constexpr uint32_t kPktInvL = kPBytes + 512;          // float[128] output factor per row (last page of a segment)
constexpr uint32_t kPktStride = kPBytes + 1024;       // 17 KiB, a multiple of 1024; all of it is copied
constexpr uint32_t kQCol = 0, kSCol0 = 320;           // S-CTA TMEM columns: Q [0,288), S buffers 320, 384
constexpr uint64_t kTimeoutNs = 500ull * 1000 * 1000;
constexpr float kLn2 = 0.69314718055994530942f;

// Layout of the two cache formats.
// bf16 cache: the S-CTA's page stage holds 64 tokens x 576 dims as 9 chunks of 64 dims,
// the O-CTA's the 512 value dims as 8 chunks; two pages in flight on each side.
// FP8 (E4M3) cache, 576 bytes a token: the S-CTA's stage holds dims 0..511 as 4 chunks of
// 128 and the 64 RoPE dims in a fifth chunk whose upper half the TMA fills with zeros,
// the O-CTA's the 512 value dims as 4 chunks; four pages in flight on each side.
// A chunk is 64 rows of 128 bytes with the 128-byte swizzle in both formats, so the
// MMA operand descriptors are the same; an FP8 MMA step covers K = 32 instead of 16.
template <bool F8>
struct Cfg {
  static constexpr int kKStages = F8 ? 4 : 2;         // S-CTA: pages in flight
  static constexpr int kVStages = F8 ? 4 : 2;         // O-CTA: pages in flight (its loads hit L2)
  static constexpr uint32_t kKChunks = F8 ? 5 : 9;
  static constexpr uint32_t kKPartA = F8 ? 4 : 5;     // chunks 0..kKPartA-1 of a page stage are released
                                                      // and refilled as soon as QK^T is done with them
  static constexpr uint32_t kVChunks = F8 ? 4 : 8;
  static constexpr uint32_t kKStageBytes = kKChunks * kChunk;
  static constexpr uint32_t kVStageBytes = kVChunks * kChunk;
  static constexpr int kQItems = F8 ? 4 : 2;          // q blocks per segment: 128 bf16 rows in blocks of 32 or 64
  static constexpr int kQRows = 128 / kQItems;
  static constexpr uint32_t kQItemBytes = static_cast<uint32_t>(kQRows) * kDimQK * 2;
  static constexpr int kKStep = F8 ? 32 : 16;         // K of one MMA step (32 bytes of a row either way)
  // The row maximum is rebased when it grows by more than 2^kRescaleLog2; P is taken
  // relative to 2^-kPOffset times the reference.  FP8: P < 2^(6+2) stays within E4M3's
  // range (448) while typical values stay clearer of its subnormals (below 2^-6) than
  // with no offset; a lower threshold would rebase O on many pages (with 2^4, about
  // half the pages of a 4096-token request with unit-scale q).
  static constexpr float kRescaleLog2 = F8 ? 6.0f : 8.0f;
  static constexpr float kPOffset = F8 ? 2.0f : 0.0f;
  // dynamic shared memory map (offsets from a 1024-byte aligned base)
  static constexpr uint32_t kOffStage = 0;
  static constexpr uint32_t kOffRecv = kVStages * kVStageBytes;            // O-CTA: kSlots packet receive slots
  static constexpr uint32_t kOffSend = kKStages * kKStageBytes;            // S-CTA: 2 packet staging slots
  static constexpr uint32_t kOffPm = kOffSend + 2 * kPktStride;            // S-CTA: row-max exchange [2][128]
  static constexpr uint32_t kOffLpart = kOffPm + 1024;                     // S-CTA: partial row sums [128]
  static constexpr uint32_t kOffInvL = kOffRecv + kSlots * kPktStride;     // O-CTA: output factor of the segment [128]
  static constexpr uint32_t kOffSharedO = kOffInvL + 512;
  static constexpr uint32_t kOffShared = kOffSharedO > kOffLpart + 512 ? kOffSharedO : kOffLpart + 512;  // both roles
  static constexpr uint32_t kOffEpi = kOffShared + 640;                    // O-CTA: 2 KiB transpose buffer per epilogue warp
  static constexpr uint32_t kOffRows = kOffEpi + 8 * 2048;                 // sparse: cache rows of kRowSlots pages
  static constexpr uint32_t kSmemBytes = kOffRows + kRowSlots * 64 * 4;
  static_assert(kKStages <= kMaxStages && kVStages <= kMaxStages, "barrier slots");
  static_assert(kQItemBytes <= kKStageBytes, "a q block fits a page stage");
  static_assert(kQItems <= kKStages, "the q blocks of a segment are resident together");
  static_assert(kOffLpart + 512 <= kOffShared, "S-CTA layout");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};
struct Bars {
  uint64_t full[kMaxStages];     // O: first half of V landed; S: part A of K, or a whole q block
  uint64_t empty[kMaxStages];    // O: first half of V free again; S: part A of K free again
  uint64_t full_b[kMaxStages];   // S: part B of K landed (plain arrival for a q block); O: second half of V
  uint64_t empty_b[kMaxStages];  // S: part B of K free again; O: second half of V free again
  uint64_t s_full[2];       // S-CTA: S = QK^T ready in TMEM
  uint64_t s_empty[2];      // S-CTA: S read by the softmax warps (8 arrivals)
  uint64_t q_full;          // S-CTA: Q of the segment stored in TMEM
  uint64_t credit[kSlots];  // S-CTA: the partner's receive slot is free (remote arrival)
  uint64_t p_full[kSlots];  // O-CTA: packet bytes arrived (bulk copy from the partner)
  uint64_t p_free[kSlots];  // O-CTA: PV MMAs that read a packet slot are done
  uint64_t o_full;          // O-CTA: the segment's last PV MMAs are done
  uint64_t o_free;          // O-CTA: epilogue finished reading O (8 arrivals)
  uint64_t o_sync;          // O-CTA: all PV MMAs issued so far are done (before a rescale)
  uint64_t corr_go;         // O-CTA: command for the rescale/epilogue warpgroups
  uint64_t corr_done;       // O-CTA: rescale finished (8 arrivals)
  uint64_t drain;           // both: final MMA completion
  uint64_t rows_full[kRowSlots];    // sparse: a page's 64 cache rows looked up (64 arrivals)
  uint64_t rows_empty[kRowSlots];   // sparse: every gathering warp has read them (one arrival each)
};

struct Shared {
  Bars bar;
  uint32_t tmem_base;
  volatile int abort;
  int cmd;                  // O-CTA command: 1 = rescale (slot in cmd_arg), 2 = epilogue, 3 = exit
  int cmd_arg;
};
static_assert(sizeof(Shared) <= 640, "control block");

struct Segment {
  int b, kb, ke, split;     // request, page range, split index within the request
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
    // A record that does not fit this call (metadata built for another batch, or
    // overwritten) would send the walk past the caller's buffers: report it and walk
    // nothing.  Every role reads the same record, so all of them stop alike.
    if (!done && (b >= prm.B || b_last < b || b_last >= prm.B || kb < 0 || k_end < 0 || split0 < 0)) {
      atomicCAS(prm.status, 0, MLA_ERR_DEVICE_BOUNDS);
      done = true;
    }
  }
  __device__ static int pages_of(int L) { return L > 0 ? (L + 63) / 64 : 0; }
  __device__ bool next(Segment& s) {
    while (!done) {
      if (b > b_last) { done = true; break; }
      const int nb = pages_of(__ldg(p->lens + b));
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

__device__ __noinline__ bool wait_bar_slow(Shared& sh, uint32_t bar, uint32_t parity, int* status,
                                           uint32_t cluster_ctas, bool cluster_scope) {
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
// Bounded wait.  Returns false on abort or timeout (after raising the abort).
__device__ __forceinline__ bool wait_bar(Shared& sh, uint32_t bar, uint32_t parity, int* status,
                                         uint32_t cluster_ctas, bool cluster_scope = false) {
  if (cluster_scope ? mbar_test_cluster(bar, parity) : mbar_test(bar, parity)) return true;
  return wait_bar_slow(sh, bar, parity, status, cluster_ctas, cluster_scope);
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

// L2 prefetch of what a segment of request b starts with: its q rows (rows x 576
// bf16, contiguous) and its block-table row.  Cold, these are many small loads
// that otherwise queue behind each other at every segment start.
__device__ __forceinline__ void prefetch_request(const DecodeParams& p, int b) {
  const uintptr_t q0 = reinterpret_cast<uintptr_t>(p.q + static_cast<int64_t>(b) * p.rows * 576);
  prefetch_l2(reinterpret_cast<const void*>(q0), static_cast<uint32_t>(p.rows) * 576 * 2);   // 16-byte multiple
  const uintptr_t t0 = reinterpret_cast<uintptr_t>(p.block_table + static_cast<int64_t>(b) * p.max_blocks);
  const uintptr_t t1 = t0 + static_cast<uintptr_t>(p.max_blocks) * 4;
  const uintptr_t a0 = t0 & ~uintptr_t(15), a1 = (t1 + 15) & ~uintptr_t(15);
  prefetch_l2(reinterpret_cast<const void*>(a0), static_cast<uint32_t>(a1 - a0));
}

// Whether split slot `slot` (partial output and lse) lies in the workspace, which holds
// B + num_parts slots; a slot outside it (metadata that does not fit the call) is
// recorded as a bounds error and its stores are skipped.
__device__ __forceinline__ bool split_slot_ok(const DecodeParams& p, int slot) {
  if (slot >= 0 && slot < p.B + p.num_parts) return true;
  atomicCAS(p.status, 0, MLA_ERR_DEVICE_BOUNDS);
  return false;
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

// ---------------------------------------------------------- sparse gather --
// Sparse decode ("为什么 MLA + MTP 容易吃亏？" section 6: the selected latents are
// gathered by index): page k of request b is entries [64k, 64k + 64) of its list, and
// entry e is the token at position t = indices[b][e], read through the block table
// like a dense token.  The rows are loaded by TMA row gathers (below) into the same
// swizzled layout a 64-row TMA box produces.

// The row lookups run in their own warps, ahead of the copies: a lane loads the list entry
// of its row two pages ahead and that token's block-table entry one page ahead, so that the
// two dependent loads of a page overlap instead of stalling the lookup warp between pages,
// and the ring of looked-up rows (row_lookup) keeps the lookups off the gathers' path.
constexpr int kNoEntry = INT_MIN;   // a row past the request's list: nothing to gather

// Walks the (request, page) pairs of one part in the order the kernel processes them.
struct PageIter {
  SegmentWalker w;
  Segment s;
  int k;
  bool valid;
  __device__ void init(const DecodeParams& p, int part) {
    w.init(p, part);
    valid = w.next(s);
    k = valid ? s.kb : 0;
  }
  __device__ void advance() {
    if (valid && ++k >= s.ke) {
      valid = w.next(s);
      k = valid ? s.kb : 0;
    }
  }
};

// Token position of row r of the iterator's page (list entry 64 k + r), or kNoEntry.
__device__ __forceinline__ int sparse_entry(const DecodeParams& p, const PageIter& it, int r, bool active) {
  if (!it.valid || !active) return kNoEntry;
  const int e = it.k * 64 + r;
  if (r >= 64 || e >= __ldg(p.lens + it.s.b)) return kNoEntry;
  if (e >= p.idx_stride) {   // a list longer than its row of indices: reported, not read
    atomicCAS(p.status, 0, MLA_ERR_DEVICE_BOUNDS);
    return kNoEntry;
  }
  return __ldg(p.indices + static_cast<int64_t>(it.s.b) * p.idx_stride + e);
}
// Block-table entry of token t of request b (checked by sparse_address), or -1 when t
// cannot be looked up.
__device__ __forceinline__ int sparse_block(const DecodeParams& p, int b, int t) {
  if (t == kNoEntry || t < 0 || t / kPageTokens >= p.max_blocks) return -1;
  return __ldg(p.block_table + static_cast<int64_t>(b) * p.max_blocks + t / kPageTokens);
}
// Address of token t's cached row (bf16: 1152 bytes; FP8: 576) given its block-table
// entry, or nullptr: past the list, or a bad entry -- a token outside [0, seqlens[b]), a
// page past the table's width or outside [0, num_blocks) -- which is recorded as a bounds
// error and not gathered.  The gather copies bytes, so the row is handed on untyped.
template <bool F8>
__device__ __forceinline__ const __nv_bfloat16* sparse_address(const DecodeParams& p, int b, int t, int blk) {
  if (t == kNoEntry) return nullptr;
  if (t < 0 || t >= __ldg(p.seqlens + b) || t / kPageTokens >= p.max_blocks || blk < 0 || blk >= p.num_blocks) {
    atomicCAS(p.status, 0, MLA_ERR_DEVICE_BOUNDS);
    return nullptr;
  }
  const int64_t row = static_cast<int64_t>(blk) * kPageTokens + t % kPageTokens;
  return reinterpret_cast<const __nv_bfloat16*>(reinterpret_cast<const uint8_t*>(p.kv) +
                                                row * (F8 ? kDimQK : 2 * kDimQK));
}

// One lookup lane's lookups: (b0, t0, blk0) for the page being looked up, (b1, t1)
// for the next one; `ahead` walks two pages ahead.
template <bool F8>
struct RowLookahead {
  PageIter ahead;
  int b0, t0, blk0, b1, t1, r;
  bool active;
  __device__ void init(const DecodeParams& p, int part, int row, bool act) {
    r = row;
    active = act;
    ahead.init(p, part);
    b0 = ahead.valid ? ahead.s.b : 0;
    t0 = sparse_entry(p, ahead, r, active);
    ahead.advance();
    blk0 = sparse_block(p, b0, t0);
    b1 = ahead.valid ? ahead.s.b : 0;
    t1 = sparse_entry(p, ahead, r, active);
    ahead.advance();
  }
  // The current page's row address; issues the next page's block-table load and the
  // list-entry load two pages ahead, then moves on by one page.
  __device__ const __nv_bfloat16* step(const DecodeParams& p) {
    const __nv_bfloat16* mine = sparse_address<F8>(p, b0, t0, blk0);
    const int blk1 = sparse_block(p, b1, t1);
    const int b2 = ahead.valid ? ahead.s.b : 0;
    const int t2 = sparse_entry(p, ahead, r, active);
    ahead.advance();
    b0 = b1, t0 = t1, blk0 = blk1, b1 = b2, t1 = t2;
    return mine;
  }
};

// ------------------------------------------------------ sparse gather by TMA --
// The sparse decode gathers a page's 64 rows by TMA, four rows per tile::gather4 load over a
// 2-D view of the cache ([cache row][576 values], a box one chunk wide and one row high: 64
// bf16 values, or 128 E4M3 codes).  The load writes its four 128-byte rows at 128-byte steps
// and swizzles each by its own shared-memory address, so 16 loads per chunk (destinations 512
// bytes apart) fill the chunk in the layout a 64-row box produces.  Two lookup warps per CTA
// find every page's rows ahead of the loads (row_lookup), and four gathering warps
// (gather_slot) take them from a ring in shared memory; four lanes of each load its four groups
// of four rows, chunk by chunk.  A row
// past the request's list, or one whose lookup fails the bounds checks (reported as a bounds
// error), loads cache row 0, which is always in range: the softmax masks it by its list
// position.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x,
                                            const int (&r)[4]) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]),
         "r"(bar)
      : "memory");
}
// kGatherSlots warps gather a page: slot gs loads rows [16 gs, 16 gs + 16), its lanes 0..3 one
// group of four rows each.  Each slot arrives once on a stage's barrier with the bytes of its own
// loads, and drains its own loads before the CTA exits.
constexpr int kGatherSlots = 4;
template <bool IsS>
__device__ __forceinline__ int gather_slot(int warp) {   // S-CTA: warps 0, 2, 3, 12; O-CTA: 0, 3, 12, 13
  if (warp == 0) return 0;
  if (IsS) return warp == 2 ? 1 : warp == 3 ? 2 : warp == 12 ? 3 : -1;
  return warp == 3 ? 1 : warp == 12 ? 2 : warp == 13 ? 3 : -1;
}
// Two lookup warps per CTA find the cache rows of every page ahead of the gathers: warp h looks
// up rows [32 h, 32 h + 32) (RowLookahead, one row per lane) and stores their row numbers in a
// ring of kRowSlots pages in shared memory.  The gathering warps only read them, so the lookups'
// dependent loads never stall the warps that issue the TMA loads.
template <bool IsS>
__device__ __forceinline__ int lookup_half(int warp) {   // S-CTA: warps 13, 14; O-CTA: 14, 15
  return IsS ? (warp == 13 ? 0 : warp == 14 ? 1 : -1) : (warp == 14 ? 0 : warp == 15 ? 1 : -1);
}
// Cache row of a looked-up address (row 0 for none: always in range, and masked by the softmax).
template <bool F8>
__device__ __forceinline__ int cache_row(const DecodeParams& p, const __nv_bfloat16* row) {
  return row ? static_cast<int>((reinterpret_cast<const uint8_t*>(row) - reinterpret_cast<const uint8_t*>(p.kv)) /
                                (F8 ? kDimQK : 2 * kDimQK))
             : 0;
}
__device__ __forceinline__ void st_shared_s32(uint32_t a, int v) {
  asm volatile("st.shared.b32 [%0], %1;" :: "r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_shared_s32(uint32_t a) {
  int v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
template <bool F8>
__device__ void row_lookup(const DecodeParams& p, Shared& sh, uint32_t smem, int part, uint32_t cl, int half) {
  using C = Cfg<F8>;
  const int lane = threadIdx.x & 31;
  RowLookahead<F8> look;
  look.init(p, part, 32 * half + lane, true);
  SegmentWalker w;
  w.init(p, part);
  Segment s;
  uint32_t T = 0;
  while (w.next(s)) {
    for (int k = s.kb; k < s.ke; ++k, ++T) {
      const int row = cache_row<F8>(p, look.step(p));   // page k of request s.b (the walks agree)
      const uint32_t slot = T % kRowSlots, ph = (T / kRowSlots) & 1;
      if (!warp_wait(sh, smem_u32(&sh.bar.rows_empty[slot]), ph ^ 1, p.status, cl)) return;
      st_shared_s32(smem + C::kOffRows + (slot * 64 + 32 * half + lane) * 4, row);
      mbar_arrive(smem_u32(&sh.bar.rows_full[slot]));
    }
  }
}
// Page T's group of four cache rows of lane `lane` of gathering slot gs (meaningful for lanes
// 0..3: rows 16 gs + 4 lane .. + 3).  Waits for the lookups, reads the rows and hands the ring
// slot back.  False on abort or timeout.
template <bool F8>
__device__ __forceinline__ bool take_rows(const DecodeParams& p, Shared& sh, uint32_t smem, uint32_t cl, uint32_t T,
                                          int gs, int lane, int (&r)[4]) {
  using C = Cfg<F8>;
  const uint32_t slot = T % kRowSlots, ph = (T / kRowSlots) & 1;
  if (!warp_wait(sh, smem_u32(&sh.bar.rows_full[slot]), ph, p.status, cl)) return false;
  const uint32_t src = smem + C::kOffRows + (slot * 64 + 16 * gs + 4 * (lane & 3)) * 4;
#pragma unroll
  for (int j = 0; j < 4; ++j) r[j] = ld_shared_s32(src + j * 4);
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&sh.bar.rows_empty[slot]));
  return true;
}

// Gathering slot gs of the S-CTA, sparse decode: the q blocks (slot 0, TMA
// boxes; the other slots only arrive) and its rows of every page (tile::gather4), part A
// (chunks 0..kKPartA-1) and part B as in the dense producer.
template <bool F8>
__device__ void s_producer_gather(const DecodeParams& p, const KvMaps* maps, Shared& sh, uint32_t smem, int part,
                                  uint32_t cl, int rb, bool withhold, int gs) {
  using C = Cfg<F8>;
  constexpr int kX = F8 ? 128 : 64;   // elements of a chunk's row
  const int lane = threadIdx.x & 31;
  SegmentWalker w;
  w.init(p, part);
  Segment s;
  uint32_t i = 0;
  int issued[C::kKStages], issued_b[C::kKStages];
  uint32_t issued_phase[C::kKStages], issued_phase_b[C::kKStages];
  for (int j = 0; j < C::kKStages; ++j) issued[j] = 0, issued_phase[j] = 0, issued_b[j] = 0, issued_phase_b[j] = 0;
  bool ok = true;
  uint32_t T = 0;   // pages
  while (ok && w.next(s)) {
    const int qrow0 = s.b * p.rows + rb * 128;
    for (int j = 0; j < C::kQItems && ok; ++j, ++i) {
      const uint32_t st = i % C::kKStages, ph = (i / C::kKStages) & 1;
      if (!warp_wait(sh, smem_u32(&sh.bar.empty[st]), ph ^ 1, p.status, cl) ||
          !warp_wait(sh, smem_u32(&sh.bar.empty_b[st]), ph ^ 1, p.status, cl)) {
        ok = false;
        break;
      }
      // Every arrival of this slot is recorded for the exit drain: the drain waits for the
      // phase of the slot's latest arrival on a stage's barrier, which the barrier cannot have
      // passed by more than one phase (an older phase's parity could alias the current one).
      const bool arrives = gs != 0 || !(withhold && i == 0);   // test hook: q block 0 never arrives
      if (lane == 0) {
        mbar_arrive(smem_u32(&sh.bar.full_b[st]));   // a q block lands whole; its second half needs no bytes
        const uint32_t full = smem_u32(&sh.bar.full[st]);
        if (gs != 0) {
          mbar_arrive(full);
        } else if (arrives) {
          mbar_arrive_expect_tx(full, C::kQItemBytes);
          tma_load_3d(smem + C::kOffStage + st * C::kKStageBytes, &maps->q, full, 0, qrow0 + C::kQRows * j, 0);
        }
      }
      issued_b[st] = 1, issued_phase_b[st] = ph;
      if (arrives) issued[st] = 1, issued_phase[st] = ph;
    }
    for (int k = s.kb; k < s.ke && ok; ++k, ++i, ++T) {
      const uint32_t st = i % C::kKStages, ph = (i / C::kKStages) & 1;
      const uint32_t stage = smem + C::kOffStage + st * C::kKStageBytes;
      int r[4];
      if (!take_rows<F8>(p, sh, smem, cl, T, gs, lane, r)) { ok = false; break; }
      if (!warp_wait(sh, smem_u32(&sh.bar.empty[st]), ph ^ 1, p.status, cl)) { ok = false; break; }
      const uint32_t full = smem_u32(&sh.bar.full[st]);
      if (lane == 0) mbar_arrive_expect_tx(full, 4u * 512u * C::kKPartA);
      __syncwarp();
      if (lane < 4)
#pragma unroll
        for (int c = 0; c < static_cast<int>(C::kKPartA); ++c)
          tma_gather4(stage + c * kChunk + (4 * gs + lane) * 512, &maps->g4, full, c * kX, r);
      issued[st] = 1, issued_phase[st] = ph;
      if (!warp_wait(sh, smem_u32(&sh.bar.empty_b[st]), ph ^ 1, p.status, cl)) { ok = false; break; }
      const uint32_t full_b = smem_u32(&sh.bar.full_b[st]);
      if (lane == 0) mbar_arrive_expect_tx(full_b, 4u * 512u * (C::kKChunks - C::kKPartA));
      __syncwarp();
      // (FP8: the RoPE chunk is bytes 512..639 of a row, 576..639 filled with zeros, as in the
      // dense loads: the MMAs never read that half)
      if (lane < 4)
#pragma unroll
        for (int c = C::kKPartA; c < static_cast<int>(C::kKChunks); ++c)
          tma_gather4(stage + c * kChunk + (4 * gs + lane) * 512, &maps->g4, full_b, c * kX, r);
      issued_b[st] = 1, issued_phase_b[st] = ph;
    }
  }
  if (lane == 0)   // this slot's loads still in flight land before the CTA may exit
    for (int st = 0; st < C::kKStages; ++st) {
      if (issued[st]) drain_bar(smem_u32(&sh.bar.full[st]), issued_phase[st]);
      if (issued_b[st]) drain_bar(smem_u32(&sh.bar.full_b[st]), issued_phase_b[st]);
    }
  __syncwarp();
}

// Gathering slot gs of the O-CTA, sparse decode: the 512 value dims of its
// rows of every page (tile::gather4), as two halves of four chunks.
template <bool F8>
__device__ void o_producer_gather(const DecodeParams& p, const KvMaps* maps, Shared& sh, uint32_t smem, int part,
                                  uint32_t cl, int gs) {
  using C = Cfg<F8>;
  constexpr int kX = F8 ? 128 : 64;   // elements of a chunk's row
  const int lane = threadIdx.x & 31;
  SegmentWalker w;
  w.init(p, part);
  Segment s;
  uint32_t T = 0;
  int issued[C::kVStages], issued_b[C::kVStages];
  uint32_t issued_phase[C::kVStages], issued_phase_b[C::kVStages];
  for (int j = 0; j < C::kVStages; ++j) issued[j] = 0, issued_phase[j] = 0, issued_b[j] = 0, issued_phase_b[j] = 0;
  constexpr int kHalf = static_cast<int>(C::kVChunks / 2);
  bool ok = true;
  while (ok && w.next(s)) {
    for (int k = s.kb; k < s.ke && ok; ++k, ++T) {
      const uint32_t st = T % C::kVStages, ph = (T / C::kVStages) & 1;
      const uint32_t stage = smem + C::kOffStage + st * C::kVStageBytes;
      int r[4];
      if (!take_rows<F8>(p, sh, smem, cl, T, gs, lane, r)) { ok = false; break; }
      if (!warp_wait(sh, smem_u32(&sh.bar.empty[st]), ph ^ 1, p.status, cl)) { ok = false; break; }
      const uint32_t full = smem_u32(&sh.bar.full[st]);
      if (lane == 0) mbar_arrive_expect_tx(full, 4u * 512u * kHalf);
      __syncwarp();
      if (lane < 4)
#pragma unroll
        for (int c = 0; c < kHalf; ++c)
          tma_gather4(stage + c * kChunk + (4 * gs + lane) * 512, &maps->g4, full, c * kX, r);
      issued[st] = 1, issued_phase[st] = ph;
      if (!warp_wait(sh, smem_u32(&sh.bar.empty_b[st]), ph ^ 1, p.status, cl)) { ok = false; break; }
      const uint32_t full_b = smem_u32(&sh.bar.full_b[st]);
      if (lane == 0) mbar_arrive_expect_tx(full_b, 4u * 512u * kHalf);
      __syncwarp();
      if (lane < 4)
#pragma unroll
        for (int c = kHalf; c < 2 * kHalf; ++c)
          tma_gather4(stage + c * kChunk + (4 * gs + lane) * 512, &maps->g4, full_b, c * kX, r);
      issued_b[st] = 1, issued_phase_b[st] = ph;
    }
  }
  if (lane == 0)   // this slot's loads still in flight land before the CTA may exit
    for (int st = 0; st < C::kVStages; ++st) {
      if (issued[st]) drain_bar(smem_u32(&sh.bar.full[st]), issued_phase[st]);
      if (issued_b[st]) drain_bar(smem_u32(&sh.bar.full_b[st]), issued_phase_b[st]);
    }
  __syncwarp();
}

// Lane 0 of warp 0 of the O-CTA: the 512 value dims of every page, as two halves
// (bf16: chunks 0..3 and 4..7, 32 KiB each; FP8: chunks 0..1 and 2..3, 16 KiB each);
// each half is refilled as soon as the PV MMAs that read it are done.
template <bool F8>
__device__ void o_producer(const DecodeParams& p, const KvMaps* maps, Shared& sh, uint32_t smem, int part,
                           uint32_t cl) {
  using C = Cfg<F8>;
  SegmentWalker w;
  w.init(p, part);
  Segment s;
  uint32_t T = 0;
  int issued[C::kVStages], issued_b[C::kVStages];
  uint32_t issued_phase[C::kVStages], issued_phase_b[C::kVStages];
  for (int j = 0; j < C::kVStages; ++j) issued[j] = 0, issued_phase[j] = 0, issued_b[j] = 0, issued_phase_b[j] = 0;
  const uint64_t policy = l2_policy_evict_first();
  bool ok = true;
  while (ok && w.next(s)) {
    for (int k = s.kb; k < s.ke && ok; ++k, ++T) {
      const uint32_t st = T % C::kVStages, ph = (T / C::kVStages) & 1;
      const uint32_t stage = smem + C::kOffStage + st * C::kVStageBytes;
      if (!wait_bar(sh, smem_u32(&sh.bar.empty[st]), ph ^ 1, p.status, cl)) { ok = false; break; }
      const int blk = request_block(p, s.b, k);
      const uint32_t full = smem_u32(&sh.bar.full[st]);
      mbar_arrive_expect_tx(full, C::kVStageBytes / 2);
      tma_load_3d_hint(stage, &maps->c4, full, 0, blk * 64, 0, policy);
      issued[st] = 1, issued_phase[st] = ph;
      if (!wait_bar(sh, smem_u32(&sh.bar.empty_b[st]), ph ^ 1, p.status, cl)) { ok = false; break; }
      const uint32_t full_b = smem_u32(&sh.bar.full_b[st]);
      mbar_arrive_expect_tx(full_b, C::kVStageBytes / 2);
      tma_load_3d_hint(stage + C::kVStageBytes / 2, &maps->c4, full_b, 0, blk * 64, C::kVChunks / 2, policy);
      issued_b[st] = 1, issued_phase_b[st] = ph;
    }
  }
  for (int st = 0; st < C::kVStages; ++st) {   // loads still in flight land before the CTA may exit
    if (issued[st]) drain_bar(smem_u32(&sh.bar.full[st]), issued_phase[st]);
    if (issued_b[st]) drain_bar(smem_u32(&sh.bar.full_b[st]), issued_phase_b[st]);
  }
}

// ------------------------------------------------------------------ S-CTA --
// The S-CTA ring walks, per segment, the q blocks of the pair's row block (bf16: rows
// 0..63 and 64..127; FP8: four blocks of 32 rows) and then the segment's pages; ring
// item i uses stage i % kKStages.

// Lane 0 of warp 0: every ring item (a q block in one TMA box, or a page in two parts).
template <bool F8>
__device__ void s_producer(const DecodeParams& p, const KvMaps* maps, Shared& sh, uint32_t smem, int part,
                           uint32_t cl, int rb, bool withhold) {
  using C = Cfg<F8>;
  SegmentWalker w;
  w.init(p, part);
  Segment s;
  uint32_t i = 0;
  int issued[C::kKStages], issued_b[C::kKStages];
  uint32_t issued_phase[C::kKStages], issued_phase_b[C::kKStages];
  for (int j = 0; j < C::kKStages; ++j) issued[j] = 0, issued_phase[j] = 0, issued_b[j] = 0, issued_phase_b[j] = 0;
  const uint64_t policy = l2_policy_evict_first();
  bool ok = true;
  while (ok && w.next(s)) {
    const int qrow0 = s.b * p.rows + rb * 128;
    for (int j = 0; j < C::kQItems && ok; ++j, ++i) {
      const uint32_t st = i % C::kKStages, ph = (i / C::kKStages) & 1;
      if (!wait_bar(sh, smem_u32(&sh.bar.empty[st]), ph ^ 1, p.status, cl) ||
          !wait_bar(sh, smem_u32(&sh.bar.empty_b[st]), ph ^ 1, p.status, cl)) {
        ok = false;
        break;
      }
      mbar_arrive(smem_u32(&sh.bar.full_b[st]));   // a q block lands whole; its second half needs no bytes
      issued_b[st] = 1, issued_phase_b[st] = ph;
      if (withhold && i == 0) continue;   // test hook: this block never arrives
      const uint32_t full = smem_u32(&sh.bar.full[st]);
      mbar_arrive_expect_tx(full, C::kQItemBytes);
      tma_load_3d(smem + C::kOffStage + st * C::kKStageBytes, &maps->q, full, 0, qrow0 + C::kQRows * j, 0);
      issued[st] = 1, issued_phase[st] = ph;
    }
    for (int k = s.kb; k < s.ke && ok; ++k, ++i) {
      const uint32_t st = i % C::kKStages, ph = (i / C::kKStages) & 1;
      const uint32_t stage = smem + C::kOffStage + st * C::kKStageBytes;
      if (!wait_bar(sh, smem_u32(&sh.bar.empty[st]), ph ^ 1, p.status, cl)) { ok = false; break; }
      const int blk = request_block(p, s.b, k);
      const uint32_t full = smem_u32(&sh.bar.full[st]);
      mbar_arrive_expect_tx(full, C::kKPartA * kChunk);
      tma_load_3d_hint(stage, &maps->k_a, full, 0, blk * 64, 0, policy);
      issued[st] = 1, issued_phase[st] = ph;
      if (!wait_bar(sh, smem_u32(&sh.bar.empty_b[st]), ph ^ 1, p.status, cl)) { ok = false; break; }
      const uint32_t full_b = smem_u32(&sh.bar.full_b[st]);
      mbar_arrive_expect_tx(full_b, C::kKStageBytes - C::kKPartA * kChunk);
      if constexpr (F8)   // the RoPE chunk: bytes 512..639 of the row, 576..639 filled with zeros
        tma_load_2d_hint(stage + C::kKPartA * kChunk, &maps->rope, full_b, kDimV, blk * 64, policy);
      else
        tma_load_3d_hint(stage + C::kKPartA * kChunk, &maps->c4, full_b, 0, blk * 64, C::kKPartA, policy);
      issued_b[st] = 1, issued_phase_b[st] = ph;
    }
  }
  for (int st = 0; st < C::kKStages; ++st) {   // loads still in flight land before the CTA may exit
    if (issued[st]) drain_bar(smem_u32(&sh.bar.full[st]), issued_phase[st]);
    if (issued_b[st]) drain_bar(smem_u32(&sh.bar.full_b[st]), issued_phase_b[st]);
  }
}

// Warp 1 of the S-CTA; all 32 lanes run the loop, one elected lane issues.
// bf16: 36 steps of K = 16 (9 chunks x 4), Q in TMEM columns [0, 288).
// FP8: Q is held as two E4M3 terms, hi in columns [0, 144) and lo in [144, 288)
// (S = Q_hi K^T + Q_lo K^T, one accumulator); 36 steps of K = 32: chunks 0..3 x 4 steps
// x {hi, lo}, then the RoPE chunk's 2 steps x {hi, lo}.
template <bool sparse, bool F8>
__device__ void s_cta_mma(const DecodeParams& p, Shared& sh, uint32_t smem, int part, uint32_t cl) {
  using C = Cfg<F8>;
  SegmentWalker w;
  w.init(p, part);
  Segment s;
  uint32_t i = 0, T = 0, seg = 0;
  const uint32_t tmem = sh.tmem_base;
  constexpr uint32_t idesc = F8 ? idesc_e4m3_f32(128, 64, 0, 0) : idesc_bf16_f32(128, 64, 0, 0);
  // one QK^T step: chunk c, 32-byte step j within its rows, Q term x (FP8 only)
  auto step = [&](uint32_t d, uint32_t kstage, int c, int j, int x, uint32_t acc) {
    const uint64_t bdesc = smem_desc_sw128(kstage + c * kChunk + j * 32, 16, 1024);
    if constexpr (F8)
      mma_f8_ts_warp(d, tmem + kQCol + x * 144 + c * 32 + j * 8, bdesc, idesc, acc);
    else
      mma_bf16_ts_warp(d, tmem + kQCol + c * 32 + j * 8, bdesc, idesc, acc);
  };
  bool ok = true, any = false;
  while (ok && w.next(s)) {
    i += C::kQItems;   // the q blocks are consumed by the softmax warps
    if (!warp_wait(sh, smem_u32(&sh.bar.q_full), seg & 1, p.status, cl)) break;
    for (int k = s.kb; k < s.ke; ++k, ++T, ++i) {
      const uint32_t st = i % C::kKStages, ph = (i / C::kKStages) & 1;
      const uint32_t sb = T & 1, sph = (T >> 1) & 1;
      if (!warp_wait(sh, smem_u32(&sh.bar.full[st]), ph, p.status, cl)) { ok = false; break; }
      if (!warp_wait(sh, smem_u32(&sh.bar.s_empty[sb]), sph ^ 1, p.status, cl)) { ok = false; break; }
      tc_fence_after();
      const uint32_t kstage = smem + C::kOffStage + st * C::kKStageBytes;
      const uint32_t d = tmem + kSCol0 + sb * 64;
      constexpr int kTerms = F8 ? 2 : 1;
#pragma unroll
      for (int c = 0; c < static_cast<int>(C::kKPartA); ++c)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int x = 0; x < kTerms; ++x) step(d, kstage, c, j, x, (c | j | x) ? 1u : 0u);
      mma_commit_warp(smem_u32(&sh.bar.empty[st]));   // part A may be refilled
      if (!warp_wait(sh, smem_u32(&sh.bar.full_b[st]), ph, p.status, cl)) { ok = false; break; }
      tc_fence_after();
      if constexpr (F8) {
#pragma unroll
        for (int j = 0; j < 2; ++j)   // dims 512..575: the first 64 bytes of the RoPE chunk
#pragma unroll
          for (int x = 0; x < 2; ++x) step(d, kstage, 4, j, x, 1u);
      } else {
#pragma unroll
        for (int c = C::kKPartA; c < 9; ++c)
#pragma unroll
          for (int j = 0; j < 4; ++j) step(d, kstage, c, j, 0, 1u);
      }
      mma_commit_warp(smem_u32(&sh.bar.empty_b[st]));
      mma_commit_warp(smem_u32(&sh.bar.s_full[sb]));
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

__device__ __forceinline__ float max32(const float (&x)[32]) {
  float m[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) m[i] = fmaxf(x[2 * i], x[2 * i + 1]);
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
  return m[0];
}

// bf16 cache: row r's q values into TMEM columns [0, 288), 2 per column.  `qrow` is
// the address of the row's first 128 bytes in its q block (chunks of kQRows rows x 128 B);
// thread (wg, r) moves dims [288 wg, 288 wg + 288) (36 16-byte units).
__device__ __forceinline__ void copy_q_to_tmem(uint32_t qrow, uint32_t chunk_bytes, uint32_t tmem_lane, int wg, int rl) {
#pragma unroll
  for (int c = 0; c < 9; ++c) {          // 9 groups of 4 units = 16 TMEM columns
    uint32_t v[16];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int u = wg * 36 + c * 4 + j;   // unit over the 576 dims: chunk u / 8, unit u % 8
      const uint4 x = ld_shared_v4(qrow + (u >> 3) * chunk_bytes + (((u & 7) ^ (rl & 7)) << 4));
      v[4 * j] = x.x, v[4 * j + 1] = x.y, v[4 * j + 2] = x.z, v[4 * j + 3] = x.w;
    }
    tmem_st16(tmem_lane + kQCol + wg * 144 + c * 16, v);
  }
}

// FP8 cache: row r's q values as two E4M3 terms, 4 values per TMEM column.  sc is the
// power of two that puts max|q| over the row in (224, 448]; hi = e4m3(q sc) goes to
// columns [0, 144) and lo = e4m3(q sc - hi) to [144, 288).  A bf16 value has 8
// significant bits: hi keeps the top 4 and the remainder, a multiple of q's last bit
// no larger than 8 of them, fits lo exactly, so hi + lo = q sc and QK^T is exact up to
// fp32 accumulation (values below ~2^-5 after scaling may lose their last bits).  One
// E4M3 term alone (2^-4 relative) would move the scores too much.  With two warpgroups
// thread (wg, r) converts dims [288 wg, 288 wg + 288) and the two agree on the row's
// maximum through pm_mine / pm_other (named barrier 1); with one, thread r converts the
// whole row.  Returns 1 / sc.
template <int kWG>
__device__ __forceinline__ float copy_q_to_tmem_f8(uint32_t qrow, uint32_t chunk_bytes, uint32_t tmem_lane, int wg,
                                                   int rl, uint32_t pm_mine, uint32_t pm_other) {
  constexpr int kUnits = 72 / kWG;        // 16-byte units (8 bf16 values) of the row per thread
  const int u0 = wg * 36;
  auto unit = [&](int u) { return ld_shared_v4(qrow + (u >> 3) * chunk_bytes + (((u & 7) ^ (rl & 7)) << 4)); };
  auto amax2 = [](float m, uint32_t w) { return fmaxf(m, fmaxf(fabsf(bf16_lo(w)), fabsf(bf16_hi(w)))); };
  float amax = 0.f;
#pragma unroll 4
  for (int j = 0; j < kUnits; ++j) {
    const uint4 x = unit(u0 + j);
    amax = amax2(amax2(amax2(amax2(amax, x.x), x.y), x.z), x.w);
  }
  if constexpr (kWG == 2) {
    asm volatile("st.shared.f32 [%0], %1;" :: "r"(pm_mine), "f"(amax) : "memory");
    named_bar_sync(1, 256);
    amax = fmaxf(amax, ld_shared_f32(pm_other));
  }
  const float t = amax > 0.f ? fminf(448.f / amax, 0x1p100f) : 1.f;
  const float sc = __uint_as_float(__float_as_uint(t) & 0x7F800000u);   // 2^floor(log2 t)
#pragma unroll 1
  for (int c = 0; c < kUnits / 4; ++c) {   // 4 units = 32 dims = 8 columns of each term
    uint32_t hi[8], lo[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 x = unit(u0 + c * 4 + j);
      const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int e = 0; e < 2; ++e) {      // dims 4e..4e+3 of the unit -> one column
        const float v0 = bf16_lo(wv[2 * e]) * sc, v1 = bf16_hi(wv[2 * e]) * sc;
        const float v2 = bf16_lo(wv[2 * e + 1]) * sc, v3 = bf16_hi(wv[2 * e + 1]) * sc;
        const uint32_t h01 = cvt_e4m3x2(v0, v1), h23 = cvt_e4m3x2(v2, v3);
        const float2 f01 = e4m3x2_to_float2(h01), f23 = e4m3x2_to_float2(h23);
        hi[2 * j + e] = h01 | (h23 << 16);
        lo[2 * j + e] = cvt_e4m3x2(v0 - f01.x, v1 - f01.y) | (cvt_e4m3x2(v2 - f23.x, v3 - f23.y) << 16);
      }
    }
    tmem_st8(tmem_lane + kQCol + 2 * u0 + c * 8, hi);          // dims 8 u0 + 32 c: column (8 u0 + 32 c) / 4
    tmem_st8(tmem_lane + kQCol + 144 + 2 * u0 + c * 8, lo);
  }
  return 1.f / sc;
}

// Warps 4..11 of the S-CTA.  Warpgroup wg (0 or 1) handles columns [32*wg, 32*wg+32)
// of every page for its 128 rows; the two exchange row maxima and partial sums
// through shared memory and use named barrier 1 (256 threads).
template <bool sparse, bool F8>
__device__ void s_cta_softmax(const DecodeParams& p, Shared& sh, uint32_t smem, int part, uint32_t cl, int rb,
                              uint32_t peer) {
  using C = Cfg<F8>;
  // Two warpgroups, each covering 32 of a page's 64 columns.
  constexpr int kWG = 2;
  constexpr uint32_t kST = kWG * 128;      // softmax threads
  constexpr int kPieces = 2 / kWG;         // 32-column pieces per thread and page
  const int t = threadIdx.x - 128;
  const int wg = t >> 7;
  const int r = t & 127;                    // row within the block == TMEM lane
  const int wq = r >> 5, lane = r & 31;
  const int c0 = wg * 32;
  const int g = rb * 128 + r;               // row within the request: i * H + h
  const bool row_valid = g < p.rows;
  const int pos_i = row_valid ? g / p.H : 0;
  const uint32_t tmem_lane = sh.tmem_base + (static_cast<uint32_t>(wq * 32) << 16);
  const uint32_t peer_recv = map_to_rank(smem + C::kOffRecv, peer);
  const uint32_t peer_pfull0 = map_to_rank(smem_u32(&sh.bar.p_full[0]), peer);
  const uint32_t pm_mine = smem + C::kOffPm + (wg * 128 + r) * 4;
  const uint32_t pm_other = smem + C::kOffPm + ((1 - wg) * 128 + r) * 4;
  const uint32_t lpart = smem + C::kOffLpart + r * 4;
  float sl2 = p.scale_log2;                 // raw score -> log2 units (FP8: per row, set with Q)
  SegmentWalker w;
  w.init(p, part);
  Segment s;
  uint32_t i = 0, T = 0;   // ring item (q blocks and pages) and page counters
  bool ok = true;
  while (ok && w.next(s)) {
    const int L = __ldg(p.lens + s.b);   // the request's list: its tokens, or its top-k entries
    int vis = L;
    if (p.causal && row_valid && !sparse) vis = L - p.s_q + pos_i + 1;
    // sparse with causal masking: an entry is visible if its token position is below
    const int vis_pos = (sparse && p.causal) ? __ldg(p.seqlens + s.b) - p.s_q + (row_valid ? pos_i : 0) + 1 : 0;
    {   // Q of this request into TMEM (every QK^T of the previous segment is complete:
        // its last S was waited for below)
      const uint32_t qi = static_cast<uint32_t>(r / C::kQRows);   // this row's q block
      const uint32_t mine = (i + qi) % C::kKStages;
      const uint32_t mph = ((i + qi) / C::kKStages) & 1;
      const bool got = wait_bar(sh, smem_u32(&sh.bar.full[mine]), mph, p.status, cl);
      if (named_bar_or(1, kST, !got)) break;
      constexpr uint32_t kQChunk = C::kQRows * 128;   // bytes per 64-dim chunk of a q block
      const int rl = r % C::kQRows;
      const uint32_t qrow = smem + C::kOffStage + mine * C::kKStageBytes + rl * 128;
      if constexpr (F8) {
        sl2 = p.scale_log2 * p.kv_scale * copy_q_to_tmem_f8<kWG>(qrow, kQChunk, tmem_lane, wg, rl, pm_mine, pm_other);
      } else {
#pragma unroll
        for (int h = 0; h < kPieces; ++h) copy_q_to_tmem(qrow, kQChunk, tmem_lane, wg + h, rl);
      }
      tmem_wait_st();
      tc_fence_before();
      named_bar_sync(1, kST);
      if (t == 0) {
        mbar_arrive(smem_u32(&sh.bar.q_full));
        for (int j = 0; j < C::kQItems; ++j) {
          const uint32_t qs = (i + j) % C::kKStages;
          mbar_arrive(smem_u32(&sh.bar.empty[qs]));
          mbar_arrive(smem_u32(&sh.bar.empty_b[qs]));
        }
        SegmentWalker nx = w;   // the next segment's q rows and block-table row, into L2 now
        Segment ns;
        if (nx.next(ns)) prefetch_request(p, ns.b);
      }
      i += C::kQItems + static_cast<uint32_t>(s.ke - s.kb);   // ring items of this segment
    }
    float m_ref = -INFINITY, l = 0.f;   // reference maximum (log2 units) and running sum of the rows
    float l_hi = 0.f;                   // one warpgroup: the running sum of columns 32..63
    for (int k = s.kb; k < s.ke; ++k, ++T) {
      const uint32_t sb = T & 1, ph = (T >> 1) & 1;
      const uint32_t rs = T % kSlots, rph = (T / kSlots) & 1;
      // S of this page; thread 0 also makes sure that staging slot sb is free (the bulk
      // copy that used it two pages ago has read it) and that the partner's receive
      // slot rs is free (its PV of the page that used it, kSlots pages ago, is done).
      bool ok_t = wait_bar(sh, smem_u32(&sh.bar.s_full[sb]), ph, p.status, cl);
      if (t == 0 && ok_t) {
        bulk_wait_group_read<1>();
        ok_t = wait_bar(sh, smem_u32(&sh.bar.credit[rs]), rph ^ 1, p.status, cl, true);
      }
      tc_fence_after();
      float sv[32];
      // raw scores of 32 columns from column cb on; slots at or past `vis` are masked to
      // -inf (only on the last pages)
      auto load_scores = [&](int cb) {
        tmem_ld32(tmem_lane + kSCol0 + sb * 64 + cb, *reinterpret_cast<uint32_t(*)[32]>(sv));
        tmem_wait_ld();
        const int nvalid = vis - (k * 64 + cb);   // columns c < nvalid are visible
        if (nvalid < 32) {
#pragma unroll
          for (int c = 0; c < 32; ++c) sv[c] = (c < nvalid) ? sv[c] : -INFINITY;
        }
        if (sparse && p.causal) {   // token positions of these 32 columns (sparse only)
          const int32_t* ix = p.indices + static_cast<int64_t>(s.b) * p.idx_stride + k * 64 + cb;
#pragma unroll
          for (int c = 0; c < 32; ++c)   // entries past the row of indices are not read (the gather reports them)
            if (c < nvalid && k * 64 + cb + c < p.idx_stride && __ldg(ix + c) >= vis_pos) sv[c] = -INFINITY;
        }
      };
      auto release_s = [&]() {   // every column of S has been read
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.bar.s_empty[sb]));
      };
      load_scores(c0);
      float my_max = max32(sv);
      if constexpr (kWG == 1) {
        load_scores(32);
        my_max = fmaxf(my_max, max32(sv));
      }
      if constexpr (kWG == 2) {
        release_s();
        asm volatile("st.shared.f32 [%0], %1;" :: "r"(pm_mine), "f"(my_max) : "memory");
      }
      // one barrier both exchanges the row maxima and makes the abort decision uniform
      if (named_bar_or(1, kST, !ok_t)) { ok = false; break; }
      // softmax_scale > 0, so the scaled maximum is the scaled raw maximum
      const float row_max = (kWG == 2) ? fmaxf(my_max, ld_shared_f32(pm_other)) : my_max;
      const float m_new = fmaxf(m_ref, row_max * (F8 ? sl2 : p.scale_log2));
      float alpha = 1.f;
      const bool rebase = m_new > m_ref + C::kRescaleLog2;
      if (rebase) {
        alpha = fast_exp2(m_ref - m_new);       // 0 when m_ref = -inf
        m_ref = m_new;
      }
      const float neg_m = (m_ref == -INFINITY) ? 0.f : (F8 ? C::kPOffset - m_ref : -m_ref);
      const uint32_t slot = smem + C::kOffSend + sb * kPktStride;
      const uint32_t row = slot + r * 128;
      float lsum[kPieces];
#pragma unroll
      for (int h = 0; h < kPieces; ++h) {
        const int cb = c0 + 32 * h;
        if constexpr (kWG == 1) load_scores(cb);   // the second pass reads the scores again
        uint32_t pk[16];
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
        // l sums the fp32 probabilities; P goes to the MMA in bf16, or (FP8) as two E4M3
        // terms hi + lo: bytes 0..63 of the row hold hi of tokens 0..63, bytes 64..127 lo
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float e0 = fast_exp2(fmaf(sv[2 * c], F8 ? sl2 : p.scale_log2, neg_m));
          const float e1 = fast_exp2(fmaf(sv[2 * c + 1], F8 ? sl2 : p.scale_log2, neg_m));
          if constexpr (F8) {
            const uint32_t h2 = cvt_e4m3x2(e0, e1);
            const float2 hf = e4m3x2_to_float2(h2);
            const uint32_t l2 = cvt_e4m3x2(e0 - hf.x, e1 - hf.y);
            if (c & 1) pk[c >> 1] |= h2 << 16, pk[8 + (c >> 1)] |= l2 << 16;
            else pk[c >> 1] = h2, pk[8 + (c >> 1)] = l2;
          } else {
            pk[c] = pack_bf16x2(e0, e1);
          }
          ps[c & 3] += e0 + e1;
        }
        lsum[h] = (ps[0] + ps[1]) + (ps[2] + ps[3]);
        if constexpr (F8) {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int cc = cb / 16 + j;             // 16-byte chunk: tokens 16cc .. 16cc+15
            st_shared_v4(row + ((cc ^ (r & 7)) << 4), make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]));
            st_shared_v4(row + (((4 + cc) ^ (r & 7)) << 4),
                         make_uint4(pk[8 + 4 * j], pk[9 + 4 * j], pk[10 + 4 * j], pk[11 + 4 * j]));
          }
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int cc = cb / 8 + j;              // 16-byte chunk: tokens 8cc .. 8cc+7
            st_shared_v4(row + ((cc ^ (r & 7)) << 4), make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]));
          }
        }
      }
      if constexpr (kWG == 1) release_s();
      // one running sum per 32-column piece, added at the segment's end: the same
      // arithmetic as two warpgroups with one piece each
      l = l * alpha + lsum[0];
      if constexpr (kPieces == 2) l_hi = l_hi * alpha + lsum[1];
      const bool last = (k == s.ke - 1);
      if (last) {   // the row sum over both halves is needed for 1/l
        if constexpr (kWG == 2) {
          if (wg == 1) asm volatile("st.shared.f32 [%0], %1;" :: "r"(lpart), "f"(l) : "memory");
          named_bar_sync(1, kST);
          if (wg == 0) l += ld_shared_f32(lpart);
        } else {
          l += l_hi;
        }
      }
      if (wg == 0) {
        asm volatile("st.shared.f32 [%0], %1;" :: "r"(slot + kPktAlpha + r * 4), "f"(alpha) : "memory");
        if (last)   // the output factor: 1/l (FP8: kv_scale / l, the value codes' scale)
          asm volatile("st.shared.f32 [%0], %1;" :: "r"(slot + kPktInvL + r * 4),
                       "f"(l > 0.f ? (F8 ? p.kv_scale : 1.f) / l : 0.f) : "memory");
      }
      fence_proxy_async_smem();
      named_bar_sync(1, kST);
      if (t == 0) {
        bulk_copy_to_cluster(peer_recv + rs * kPktStride, slot, kPktStride, peer_pfull0 + rs * 8);
        bulk_commit_group();
      }
    }
    if (!ok) break;
    if (row_valid && wg == 0) {
      const float lse = l > 0.f ? ((F8 ? m_ref - C::kPOffset : m_ref) + log2f(l)) * kLn2 : -INFINITY;
      const int ns0 = __ldg(p.num_splits + s.b);
      const int nsplit = __ldg(p.num_splits + s.b + 1) - ns0;
      if (nsplit == 1)
        p.lse[static_cast<int64_t>(s.b) * p.rows + g] = lse;
      else if (split_slot_ok(p, ns0 + s.split))
        p.lse_part[static_cast<int64_t>(ns0 + s.split) * p.rows + g] = lse;
    }
  }
  if (t == 0) bulk_wait_group<0>();   // copies land before the CTA may exit
}

// ------------------------------------------------------------------ O-CTA --
// Warp 1 of the O-CTA (all 32 lanes; one elected lane issues the MMAs).  Per page and
// 256-column half of O: bf16, one MMA per 16 tokens; FP8, two per 32 tokens (the hi and
// the lo term of P against the same value rows).
template <bool sparse, bool F8>
__device__ void o_cta_mma(const DecodeParams& p, Shared& sh, uint32_t smem, int part, uint32_t cl) {
  using C = Cfg<F8>;
  constexpr int kHalfChunks = static_cast<int>(C::kVChunks / 2);
  constexpr int kTerms = F8 ? 2 : 1;
  const int lane = threadIdx.x & 31;
  SegmentWalker w;
  w.init(p, part);
  Segment s;
  uint32_t T = 0, seg = 0, nresc = 0;
  const uint32_t tmem = sh.tmem_base;
  constexpr uint32_t idesc = F8 ? idesc_e4m3_f32(128, 256, 0, 1) : idesc_bf16_f32(128, 256, 0, 1);
  bool ok = true, any = false;
  while (ok && w.next(s)) {
    if (seg > 0 && !warp_wait(sh, smem_u32(&sh.bar.o_free), (seg - 1) & 1, p.status, cl)) break;
    const int L = __ldg(p.lens + s.b);
    for (int k = s.kb; k < s.ke; ++k, ++T) {
      const uint32_t st = T % C::kVStages, ph = (T / C::kVStages) & 1;
      const uint32_t ps = T % kSlots, pph = (T / kSlots) & 1;
      const uint32_t vstage = smem + C::kOffStage + st * C::kVStageBytes;
      const uint32_t pkt = smem + C::kOffRecv + ps * kPktStride;
      if (lane == 0) mbar_arrive_expect_tx(smem_u32(&sh.bar.p_full[ps]), kPktStride);
      __syncwarp();
      if (!warp_wait(sh, smem_u32(&sh.bar.full[st]), ph, p.status, cl)) { ok = false; break; }
      if (!warp_wait(sh, smem_u32(&sh.bar.p_full[ps]), pph, p.status, cl, true)) { ok = false; break; }
      // tail page: zero the value rows past the sequence end up to the next MMA-step
      // boundary, so that P = 0 never meets a non-finite value in the MMA (per half)
      const int nvalid = min(64, L - k * 64);
      const int krows = (nvalid + C::kKStep - 1) & ~(C::kKStep - 1);
      auto zero_tail = [&](uint32_t half) {
        if (nvalid < krows) {
          const int nz = krows - nvalid;                           // rows to clear, < kKStep
          for (int i = lane; i < nz * kHalfChunks * 8; i += 32) {  // rows x chunks x 16-byte units
            const int row = nvalid + i / (kHalfChunks * 8), chunk = (i / 8) % kHalfChunks, u = i % 8;
            st_shared_v4(half + chunk * kChunk + row * 128 + u * 16, make_uint4(0, 0, 0, 0));
          }
          fence_proxy_async_smem();
        }
      };
      zero_tail(vstage);
      const bool last = (k == s.ke - 1);
      if (last)     // keep 1/l of the segment's rows before the slot can be reused
        st_shared_v4(smem + C::kOffInvL + lane * 16, ld_shared_v4(pkt + kPktInvL + lane * 16));
      bool need = false;
      if (k != s.kb) {   // did any row rebase its maximum on this page?
        const uint4 a = ld_shared_v4(pkt + kPktAlpha + lane * 16);
        need = __any_sync(0xffffffffu, a.x != 0x3f800000u || a.y != 0x3f800000u || a.z != 0x3f800000u ||
                                           a.w != 0x3f800000u);
      }
      __syncwarp();
      if (need) {   // scale O by alpha before adding this page
        mma_commit_warp(smem_u32(&sh.bar.o_sync));
        if (!warp_wait(sh, smem_u32(&sh.bar.o_sync), nresc & 1, p.status, cl)) { ok = false; break; }
        if (lane == 0) {
          sh.cmd = 1;
          sh.cmd_arg = static_cast<int>(ps);
          mbar_arrive(smem_u32(&sh.bar.corr_go));
        }
        __syncwarp();
        if (!warp_wait(sh, smem_u32(&sh.bar.corr_done), nresc & 1, p.status, cl)) { ok = false; break; }
        ++nresc;
      }
      __syncwarp();
      tc_fence_after();
      {
        const int ksteps = krows / C::kKStep;
        // O[:, 256 h .. 256 h + 255] += P V over the value chunks of half h; step js covers
        // tokens [kKStep js, kKStep js + kKStep) (P: 32 bytes of the row, term x at byte 64 x)
        auto pv = [&](int h, uint32_t vhalf) {
          for (int js = 0; js < ksteps; ++js)
#pragma unroll
            for (int x = 0; x < kTerms; ++x) {
              const uint64_t adesc = smem_desc_sw128(pkt + x * 64 + js * 32, 16, 1024);
              const uint64_t bdesc = smem_desc_sw128(vhalf + js * C::kKStep * 128, 8192, 1024);
              const uint32_t acc = (k == s.kb && js == 0 && x == 0) ? 0u : 1u;
              if constexpr (F8) mma_f8_ss_warp(tmem + 256 * h, adesc, bdesc, idesc, acc);
              else mma_bf16_ss_warp(tmem + 256 * h, adesc, bdesc, idesc, acc);
            }
        };
        pv(0, vstage);                                  // output columns 0..255
        mma_commit_warp(smem_u32(&sh.bar.empty[st]));   // the first half may be refilled
        if (!warp_wait(sh, smem_u32(&sh.bar.full_b[st]), ph, p.status, cl)) { ok = false; break; }
          zero_tail(vstage + C::kVStageBytes / 2);
        __syncwarp();
        tc_fence_after();
        pv(1, vstage + C::kVStageBytes / 2);            // output columns 256..511
        mma_commit_warp(smem_u32(&sh.bar.empty_b[st]));
        mma_commit_warp(smem_u32(&sh.bar.p_free[ps]));
        if (last) mma_commit_warp(smem_u32(&sh.bar.o_full));
      }
      any = true;
      __syncwarp();
      if (last && lane == 0) {
        sh.cmd = 2;
        sh.cmd_arg = static_cast<int>(seg);
        mbar_arrive(smem_u32(&sh.bar.corr_go));
      }
      __syncwarp();
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
}

// Warp 2 of the O-CTA: returns each packet slot to the S-CTA once the MMAs reading it are done.
__device__ void o_cta_forwarder(const DecodeParams& p, Shared& sh, int part, uint32_t cl, uint32_t peer) {
  SegmentWalker w;
  w.init(p, part);
  Segment s;
  uint32_t T = 0;
  const uint32_t credit0 = map_to_rank(smem_u32(&sh.bar.credit[0]), peer);
  bool ok = true;
  while (ok && w.next(s)) {
    for (int k = s.kb; k < s.ke; ++k, ++T) {
      const uint32_t ps = T % kSlots, pph = (T / kSlots) & 1;
      if (!wait_bar(sh, smem_u32(&sh.bar.p_free[ps]), pph, p.status, cl)) { ok = false; break; }
      mbar_arrive_remote(credit0 + ps * 8);
    }
  }
}

// Warps 4..11 of the O-CTA: rescale O rows, or normalise and store a finished
// segment.  Warpgroup wg owns O columns [256 wg, 256 wg + 256).
// Two warpgroups, one per 256-column half of O.
template <bool sparse, bool F8>
__device__ void o_cta_epilogue(const DecodeParams& p, Shared& sh, uint32_t smem, int part, uint32_t cl, int rb) {
  using C = Cfg<F8>;
  constexpr int kHalves = 1;   // 256-column halves of O per thread
  const int t = threadIdx.x - 128;
  const int wg = t >> 7;
  const int r = t & 127;
  const int wq = r >> 5, lane = r & 31;
  const uint32_t tmem_row = sh.tmem_base + (static_cast<uint32_t>(wq * 32) << 16);
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
      const float alpha = ld_shared_f32(smem + C::kOffRecv + arg * kPktStride + kPktAlpha + r * 4);
      tc_fence_after();
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < 256 * kHalves; c += 32) {
          const uint32_t col = tmem_row + wg * 256 + c;
          uint32_t v[32];
          tmem_ld32(col, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
          tmem_st32(col, v);
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
    const float inv_l = ld_shared_f32(smem + C::kOffInvL + r * 4);
    const int ns0 = __ldg(p.num_splits + s.b);
    const int nsplit = __ldg(p.num_splits + s.b + 1) - ns0;
    const bool final_out = (nsplit == 1);
    const bool slot_ok = final_out || split_slot_ok(p, ns0 + s.split);   // partial stores stay in the workspace
    // Stores go through the warp's transpose buffer: a thread holds one row's columns, so
    // direct stores would touch 32 rows per instruction; transposed, each store
    // instruction writes 64 contiguous bytes of 8 rows.  Buffer row x (64 B) holds
    // 16-byte unit u at ((u ^ ((x >> 1) & 3)) * 16): the 8 rows a quarter-warp stores (or
    // the 2 rows it loads) then touch 8 distinct 16-byte bank groups.
    const int g0 = rb * 128 + wq * 32;    // the warp's first row within the request
    __nv_bfloat16* const obase0 = p.out + (static_cast<int64_t>(s.b) * p.rows + g0) * 512;
    float* const pbase0 = p.o_part + (static_cast<int64_t>(ns0 + s.split) * p.rows + g0) * 512;
    const uint32_t stg = smem + C::kOffEpi + ((wg << 2) | wq) * 2048;
    const int tq = lane & 3;                // transposed: 16-byte quad tq of rows 8j + (lane >> 2)
    auto put = [&](int j, uint4 u) { st_shared_v4(stg + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4), u); };
    auto get = [&](int j) {
      const int x = 8 * j + (lane >> 2);
      return ld_shared_v4(stg + x * 64 + ((tq ^ ((x >> 1) & 3)) << 4));
    };
    // column chunk hc (32 columns) of this warpgroup's part of O, then its stores
    auto col_of = [&](int hc) { return tmem_row + (wg + hc / 256) * 256 + hc % 256; };
    auto emit = [&](int hc, const uint32_t (&v)[32]) {
      const int half = wg + hc / 256, c = hc % 256;   // column c of O's half `half`
      __nv_bfloat16* const obase = obase0 + half * 256;
      float* const pbase = pbase0 + half * 256;
      if (final_out) {   // 32 bf16 columns: 64 B per row
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint4 u;
          u.x = pack_bf16x2(__uint_as_float(v[8 * j + 0]) * inv_l, __uint_as_float(v[8 * j + 1]) * inv_l);
          u.y = pack_bf16x2(__uint_as_float(v[8 * j + 2]) * inv_l, __uint_as_float(v[8 * j + 3]) * inv_l);
          u.z = pack_bf16x2(__uint_as_float(v[8 * j + 4]) * inv_l, __uint_as_float(v[8 * j + 5]) * inv_l);
          u.w = pack_bf16x2(__uint_as_float(v[8 * j + 6]) * inv_l, __uint_as_float(v[8 * j + 7]) * inv_l);
          put(j, u);
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int x = 8 * j + (lane >> 2);
          const uint4 u = get(j);
          if (g0 + x < p.rows) *reinterpret_cast<uint4*>(obase + static_cast<int64_t>(x) * 512 + c + 8 * tq) = u;
        }
        __syncwarp();
      } else {           // fp32 partials: two passes of 16 columns (64 B per row)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int e = 16 * h + 4 * j;
            put(j, make_uint4(__float_as_uint(__uint_as_float(v[e]) * inv_l), __float_as_uint(__uint_as_float(v[e + 1]) * inv_l),
                              __float_as_uint(__uint_as_float(v[e + 2]) * inv_l), __float_as_uint(__uint_as_float(v[e + 3]) * inv_l)));
          }
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int x = 8 * j + (lane >> 2);
            const uint4 u = get(j);
            if (g0 + x < p.rows && slot_ok)
              *reinterpret_cast<uint4*>(pbase + static_cast<int64_t>(x) * 512 + c + 16 * h + 4 * tq) = u;
          }
          __syncwarp();
        }
      }
    };
    // the TMEM load of the next 32 columns is in flight while the current ones are stored
    constexpr int kSteps = 256 * kHalves;
    uint32_t va[32], vb[32];
    tmem_ld32(col_of(0), va);
#pragma unroll 1
    for (int hc = 0; hc < kSteps; hc += 64) {
      tmem_wait_ld();
      tmem_ld32(col_of(hc + 32), vb);
      emit(hc, va);
      tmem_wait_ld();
      if (hc + 64 < kSteps) {
        tmem_ld32(col_of(hc + 64), va);
      } else {   // everything read: O may be overwritten by the next segment
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.bar.o_free));
      }
      emit(hc + 32, vb);
    }
    ++seg;
    have_seg = w.next(s);
  }
}

}  // namespace

// kSparse: the pages are gathered from the top-k lists (p.indices) instead of read whole.
// kF8: the cache holds E4M3 codes with one per-tensor scale (p.kv_scale).
template <bool kSparse, bool kF8>
__global__ void __launch_bounds__(threads_of<kSparse, kF8>(), 1)
mla_decode_kernel(const __grid_constant__ KvMaps maps, const DecodeParams p) {
  using C = Cfg<kF8>;
  extern __shared__ __align__(1024) uint8_t dyn_smem[];
  const uint32_t base = smem_u32(dyn_smem);
  if (base & 1023u) {   // the layout needs a 1024-byte aligned base (no static shared memory is declared)
    if (threadIdx.x == 0) atomicCAS(p.status, 0, MLA_ERR_UNSUPPORTED);
    return;             // every CTA of the grid takes this branch alike
  }
  const uint32_t smem = base;
  Shared& sh = *reinterpret_cast<Shared*>(dyn_smem + C::kOffShared);
  const int warp = threadIdx.x >> 5;
  const uint32_t rank = cluster_ctarank();
  const uint32_t cl = 2u * static_cast<uint32_t>(p.n_rb);   // CTAs per cluster
  const int part = static_cast<int>(blockIdx.x / cl);
  const int rb = static_cast<int>(rank >> 1);
  const bool is_s = (rank & 1u) == 0;
  const uint32_t peer = rank ^ 1u;

  if (threadIdx.x == 0) {
    if (is_s) {
      prefetch_tensormap(&maps.q);
      prefetch_tensormap(&maps.k_a);
      if (kF8) prefetch_tensormap(&maps.rope);
    }
    prefetch_tensormap(&maps.c4);
    sh.abort = 0;
    sh.cmd = 0;
    // sparse: one arrival per gathering warp, each with its own bytes; dense: the producer's one
    // arrival with the expected bytes
    constexpr uint32_t kGroupWarps = 8;   // softmax / epilogue warps
    const uint32_t fills = kSparse ? static_cast<uint32_t>(kGatherSlots) : 1u;
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(smem_u32(&sh.bar.full[i]), fills);
      mbar_init(smem_u32(&sh.bar.empty[i]), 1);
      mbar_init(smem_u32(&sh.bar.full_b[i]), fills);
      mbar_init(smem_u32(&sh.bar.empty_b[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sh.bar.s_full[i]), 1);
      mbar_init(smem_u32(&sh.bar.s_empty[i]), kGroupWarps);   // one arrival per softmax warp
    }
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(smem_u32(&sh.bar.credit[i]), 1);
      mbar_init(smem_u32(&sh.bar.p_full[i]), 1);
      mbar_init(smem_u32(&sh.bar.p_free[i]), 1);
    }
    mbar_init(smem_u32(&sh.bar.q_full), 1);
    mbar_init(smem_u32(&sh.bar.o_full), 1);
    mbar_init(smem_u32(&sh.bar.o_free), kGroupWarps);            // one arrival per epilogue warp
    mbar_init(smem_u32(&sh.bar.o_sync), 1);
    mbar_init(smem_u32(&sh.bar.corr_go), 1);
    mbar_init(smem_u32(&sh.bar.corr_done), kGroupWarps);
    mbar_init(smem_u32(&sh.bar.drain), 1);
    for (int i = 0; i < kRowSlots; ++i) {
      mbar_init(smem_u32(&sh.bar.rows_full[i]), 64);              // one arrival per looked-up row
      mbar_init(smem_u32(&sh.bar.rows_empty[i]), kGatherSlots);   // one arrival per gathering warp
    }
    fence_mbar_init();
  }
  __syncwarp();
  if (warp == 0) tmem_alloc(smem_u32(&sh.tmem_base), 512);
  tc_fence_before();
  __syncthreads();
  cluster_sync();        // every barrier of the cluster is initialised before any remote use
  tc_fence_after();
  griddep_wait();        // the metadata, q and the cache are complete from here on
  if (threadIdx.x == 0 && is_s && rb == 0) {   // first request's q rows and block-table row
    const int b0 = p.meta[part * 8];
    if (b0 >= 0) prefetch_request(p, b0);
  }

  // sparse: two warps look up the listed rows (row_lookup) and four load them by TMA
  // (s_producer_gather / o_producer_gather)
  if (is_s) {
    if (kSparse && gather_slot<true>(warp) >= 0) {
      s_producer_gather<kF8>(p, &maps, sh, smem, part, cl, rb, p.withhold_first_load != 0, gather_slot<true>(warp));
    } else if (!kSparse && warp == 0) {
      if ((threadIdx.x & 31) == 0) s_producer<kF8>(p, &maps, sh, smem, part, cl, rb, p.withhold_first_load != 0);
    } else if (warp == 1) {
      s_cta_mma<kSparse, kF8>(p, sh, smem, part, cl);
    } else if (warp >= 4 && warp < 12) {
      s_cta_softmax<kSparse, kF8>(p, sh, smem, part, cl, rb, peer);
    } else if (kSparse && lookup_half<true>(warp) >= 0) {
      row_lookup<kF8>(p, sh, smem, part, cl, lookup_half<true>(warp));
    }
  } else {
    if (kSparse && gather_slot<false>(warp) >= 0) {
      o_producer_gather<kF8>(p, &maps, sh, smem, part, cl, gather_slot<false>(warp));
    } else if (!kSparse && warp == 0) {
      if ((threadIdx.x & 31) == 0) o_producer<kF8>(p, &maps, sh, smem, part, cl);
    } else if (warp == 1) {
      o_cta_mma<kSparse, kF8>(p, sh, smem, part, cl);
    } else if (warp == 2) {
      if ((threadIdx.x & 31) == 0) o_cta_forwarder(p, sh, part, cl, peer);
    } else if (warp >= 4 && warp < 12) {
      o_cta_epilogue<kSparse, kF8>(p, sh, smem, part, cl, rb);
    } else if (kSparse && lookup_half<false>(warp) >= 0) {
      row_lookup<kF8>(p, sh, smem, part, cl, lookup_half<false>(warp));
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
  cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(Cfg<false>::kSmemBytes));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(mla_decode_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(Cfg<false>::kSmemBytes));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(mla_decode_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(Cfg<true>::kSmemBytes));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(mla_decode_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(Cfg<true>::kSmemBytes));
}

// attr[0] = the cluster shape; with pdl, attr[1] = programmatic stream serialisation
// (both cache formats use the same amount of shared memory)
static_assert(Cfg<false>::kSmemBytes == Cfg<true>::kSmemBytes, "one launch shape for both formats");
static cudaLaunchConfig_t decode_config(int grid_ctas, int cluster_ctas, cudaStream_t stream,
                                        cudaLaunchAttribute* attr, bool pdl, int threads = kThreads) {
  cudaLaunchConfig_t cfg = pdl_config(dim3(static_cast<unsigned>(grid_ctas), 1, 1),
                                      dim3(static_cast<unsigned>(threads), 1, 1), Cfg<false>::kSmemBytes, stream,
                                      attr + 1);
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster_ctas);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cfg;
}

int decode_max_clusters(int cluster_ctas) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = decode_config(cluster_ctas, cluster_ctas, nullptr, attr, false);
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, mla_decode_kernel<false, false>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return clusters;
}

cudaError_t launch_decode(const KvMaps& maps, const DecodeParams& p, int cluster_ctas, cudaStream_t stream) {
  cudaLaunchAttribute attr[2];
  if (p.indices) {   // 16 warps (one CTA per SM either way: shared memory bounds it)
    static_assert(threads_of<true, true>() == threads_of<true, false>(), "one sparse launch shape");
    cudaLaunchConfig_t cfg16 = decode_config(p.num_parts * cluster_ctas, cluster_ctas, stream, attr, true,
                                             threads_of<true, true>());
    if (p.kv_fp8) return cudaLaunchKernelEx(&cfg16, mla_decode_kernel<true, true>, maps, p);
    return cudaLaunchKernelEx(&cfg16, mla_decode_kernel<true, false>, maps, p);
  }
  cudaLaunchConfig_t cfg = decode_config(p.num_parts * cluster_ctas, cluster_ctas, stream, attr, true);
  if (p.kv_fp8) return cudaLaunchKernelEx(&cfg, mla_decode_kernel<false, true>, maps, p);
  return cudaLaunchKernelEx(&cfg, mla_decode_kernel<false, false>, maps, p);
}

}  // namespace mla
