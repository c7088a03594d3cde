// Internal interface between the host ABI (mla_host.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "mla.h"

namespace mla {

constexpr int kPageTokens = 64;
constexpr int kDimQK = 576;
constexpr int kDimV = 512;
constexpr int kRowsPerPair = 128;
constexpr int kMaxPairsPerCluster = 4;
constexpr int kMetaInts = 8;            // ints per part record

// Schedule constants (the CPU restatement in the tests reads them through
// mla_schedule_params).
constexpr int kSegmentCostPages = 2;    // one segment's set-up + epilogue, in pages
constexpr int kHbmParts = 64;           // clusters that already saturate HBM
constexpr int kSplitCostPages = 12;     // estimated cost of an extra segment (q reload, partials, combine)
constexpr int kScheduleThreads = 512;
constexpr int kScheduleMaxB = 16384;    // requests per batch (the schedule keeps its prefix sums in shared memory)

struct DecodeParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kv;
  int64_t num_blocks;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* seqlens;
  // The per-request list the kernel walks in pages of 64 entries: seqlens itself
  // (dense), or the top-k list lengths (sparse: entry e of request b is the token at
  // position indices[b * idx_stride + e]; indices == nullptr for the dense decode).
  const int32_t* lens;
  const int32_t* indices;
  int64_t idx_stride;
  int B, s_q, H, rows, n_rb;
  float scale_log2;                     // softmax_scale * log2(e)
  int causal;
  const int32_t* meta;                  // [num_parts][8]
  const int32_t* num_splits;            // [B + 1]
  int num_parts;
  float* o_part;                        // [max_splits][rows][512]
  float* lse_part;                      // [max_splits][rows]
  __nv_bfloat16* out;                   // [B][rows][512]
  float* lse;                           // [B][rows]
  int* status;
  int withhold_first_load;
  // FP8 cache: kv holds E4M3 codes (576 bytes a token) and a cached value is its code's
  // value times kv_scale.
  int kv_fp8 = 0;
  float kv_scale = 1.f;
};

// Tensor maps of the decode kernel.  Every box lands in the swizzled (128-byte),
// chunk-major shared-memory layout the MMAs read: chunks of 128-byte rows.
// bf16 cache: the cache and q are both viewed as [chunk 0..8][row][64 dims]: dim 0 =
// 64 dims of a chunk (128 B, contiguous), dim 1 = rows (stride 1152 B: cache tokens,
// or q rows b * s_q * H + i * H + h), dim 2 = chunk (stride 128 B); k_a = chunks 0..4
// of a page (40 KiB), c4 = four chunks (32 KiB: K chunks 5..8, V chunks 0..3 or 4..7),
// q = 64 q rows (72 KiB).
// FP8 cache: the cache is viewed as [chunk 0..3][row][128 codes] (row stride 576 B):
// k_a = chunks 0..3 of a page (32 KiB), c4 = two chunks (16 KiB: V chunks 0..1 or
// 2..3); rope = the cache as [row][576 codes], read as a 128-code box at code 512 (the
// 64 RoPE codes, the rest of the box filled with zeros); q = 32 q rows (36 KiB).
struct KvMaps {
  CUtensorMap k_a;
  CUtensorMap c4;
  CUtensorMap q;
  CUtensorMap rope;   // FP8 cache only
  CUtensorMap g4;     // bf16 cache as [cache row][576 dims], box 64 dims x 1 row (tile::gather4 loads)
};
// Encodes the maps for a bf16 cache of num_blocks pages and q_rows rows of q; false on
// failure.
bool encode_kv_maps(PFN_cuTensorMapEncodeTiled_v12000 encode, KvMaps* maps, const void* kv_cache, int64_t num_blocks,
                    const void* q, int64_t q_rows);
// The same for an FP8 (E4M3) cache.
bool encode_kv_maps_fp8(PFN_cuTensorMapEncodeTiled_v12000 encode, KvMaps* maps, const void* kv_cache,
                        int64_t num_blocks, const void* q, int64_t q_rows);

// Device address of the kernels' status word on the current device (set-up on
// first use); nullptr on error.
int* device_status_word();

// Launch configuration shared by every kernel of the library: programmatic stream
// serialisation, so that a kernel's set-up overlaps the tail of the kernel before it
// on the stream (each kernel waits on griddepcontrol before its first global access).
inline cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                     cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Launchers (defined next to their kernels).
cudaError_t decode_set_attributes();
int decode_max_clusters(int cluster_ctas);            // occupancy query; 0 on error
cudaError_t launch_decode(const KvMaps& maps, const DecodeParams& p, int cluster_ctas, cudaStream_t stream);

cudaError_t launch_schedule(const int32_t* seqlens, int B, int num_parts, int fixed_cost, int hbm_parts,
                            int split_cost, int32_t* meta, int32_t* num_splits, cudaStream_t stream);
// max_splits: partial slots in the workspace (B + num_parts); split offsets beyond it
// are reported as MLA_ERR_DEVICE_BOUNDS in *status instead of read.
cudaError_t launch_combine(const float* o_part, const float* lse_part, const int32_t* num_splits, int B, int rows,
                           int max_splits, __nv_bfloat16* out, float* lse, int* status, cudaStream_t stream);

struct BmmParams {
  __nv_bfloat16* out;
  int64_t out_row_stride;   // elements between tokens n
  int64_t out_head_stride;  // elements between heads h
  int N;                    // tokens
  int H;
  int* status;
  const __nv_bfloat16* pe;  // optional: copied into out[n, h, 512:576] by the first column tile
  int64_t pe_row_stride;
  // optional RoPE of the copied q_pe: positions [N] and, per pair j of the 64 values,
  // the inverse frequency theta^(-2j/64) as a float pair (hi + lo); 2*pi as a float
  // pair for the reduction of the angle
  const int32_t* positions;
  float rope_hi[32], rope_lo[32];
  float two_pi_hi, two_pi_lo;
  // the weights [H][K * N] (bf16 kernels): each head's matrix is prefetched into L2 before
  // the kernel waits for the previous one (a prefetch only; the TMA loads come after)
  const __nv_bfloat16* w = nullptr;
  // optional (bf16 absorption): one more CTA of the grid computes the split schedule
  // (the rule and the bytes of mla_decode_metadata) for sched_B requests and sched_parts
  // parts into sched_meta; its prefix sums use the CTA's shared memory (kAbsorbPlanMaxB)
  const int32_t* sched_seqlens = nullptr;
  int32_t* sched_meta = nullptr;
  int sched_B = 0, sched_parts = 0, sched_fixed = 0, sched_hbm = 0, sched_split = 0;
};
constexpr int kAbsorbPlanMaxB = 8000;   // (B + 1) * 8 + B * 4 bytes within the absorption's 97 KB
cudaError_t bmm_set_attributes();
// absorb: K = 128 -> 512 columns; unabsorb: K = 512 -> 128 columns
cudaError_t launch_bmm(bool absorb, const CUtensorMap& a_map, const CUtensorMap& w_map, const CUtensorMap& o_map,
                       const BmmParams& p, cudaStream_t stream);

// FP8 projections: x (bf16) quantized per tensor on the fly, E4M3 weights stored transposed
// ([H, J, K], K contiguous) with one per-tensor scale.  `partials` (kAmaxParts floats of
// caller workspace) receives the partial maxima of |x| that the bmm kernel reduces.
constexpr int kAmaxParts = 128;
struct BmmFp8Params {
  BmmParams base;           // output, strides, N, H, status, the optional q_pe copy / RoPE
  const float* partials;    // [kAmaxParts]
  const uint8_t* w;         // [H, J, K] E4M3 codes
  int J;                    // output columns per head (512: absorption, 128: un-absorption)
  float w_scale;
};
cudaError_t bmm_fp8_set_attributes();
cudaError_t launch_bmm_fp8(bool absorb, const __nv_bfloat16* x, int64_t x_row_stride, int K, const CUtensorMap& x_map,
                           const CUtensorMap& w_map, const CUtensorMap& o_map, const BmmFp8Params& p, float* partials,
                           cudaStream_t stream);

// Chunked extend on the expanded path: one chunk [c0, c0 + n) of a request's cache.
struct ExtendParams {
  const int32_t* block_row;     // the request's block-table row (device)
  int64_t num_blocks;
  int c0, n, cap;               // chunk start (a multiple of 64), its tokens, Kx / Vx rows
  int T, H, qpos0;              // new tokens, heads, position of new token 0 (seqlen - T)
  float scale_log2;             // softmax_scale * log2(e)
  __nv_bfloat16* kx;            // [H, cap, 128] expanded keys (no RoPE part), head-major
  __nv_bfloat16* vx;            // [H, cap, 128] expanded values, head-major
  float* acc_o;                 // [T, H, 128] running merged output (fp32)
  float* acc_lse;               // [T, H] running merged lse
  int first, last;              // the first / last chunk of the call
  int defer_wait;               // expansion: griddepcontrol.wait at its end, not its start (below)
  __nv_bfloat16* out;           // [T, H, 128] bf16 (written by the last chunk)
  float* lse;                   // [T, H] (written by the last chunk)
  int* status;
};
struct ExtendMaps {
  CUtensorMap c;                // cache [chunk 0..8][row][64 dims], box 64 x 64 rows x 1 chunk
  CUtensorMap wk;               // W_UK as [H * 128 rows][512], box 64 x 128
  CUtensorMap wv;               // W_UV as [H * 512 rows][128], box 64 x 64
  CUtensorMap qn;               // q_nope [128, H, T], box 64 x 1 x 128
  CUtensorMap qp;               // q_pe [64, H, T], box 64 x 1 x 128
  CUtensorMap kx[2], vx[2];     // the two Kx / Vx buffers as [128, cap, H], box 64 x 64 x 1
  CUtensorMap kr;               // the cache view of c, k^R = chunk 8
};
cudaError_t extend_set_attributes();
cudaError_t launch_extend_chunk(const ExtendMaps& maps, const ExtendParams& p, int buf, cudaStream_t stream);

}  // namespace mla
