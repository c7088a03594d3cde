// Host side of the C ABI in include/mla.h: argument checks, TMA descriptors,
// launch configuration.  No device memory is allocated here.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <cmath>
#include <mutex>

#include "mla_kernels.h"

namespace mla {
namespace {

__device__ int g_device_status;   // written by the kernels, read by mla_get_device_status

int g_withhold_first_load = 0;

constexpr int kMaxDevices = 64;
struct DeviceState {
  bool ready = false;
  int* status = nullptr;
  int sm_count = 0;
  int parts[kMaxPairsPerCluster + 1] = {0, 0, 0, 0, 0};
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// One-time per-device set-up: kernel attributes, status-word address.
mla_status_t device_state(int dev, DeviceState** out) {
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return MLA_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_device_status) != cudaSuccess) return MLA_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MLA_ERR_CUDA;
    if (decode_set_attributes() != cudaSuccess) return MLA_ERR_CUDA;
    if (bmm_set_attributes() != cudaSuccess) return MLA_ERR_CUDA;
    if (bmm_fp8_set_attributes() != cudaSuccess) return MLA_ERR_CUDA;
    if (extend_set_attributes() != cudaSuccess) return MLA_ERR_CUDA;
    for (int n = 1; n <= kMaxPairsPerCluster; ++n) d.parts[n] = decode_max_clusters(2 * n);
    d.ready = true;
  }
  *out = &d;
  return MLA_OK;
}

mla_status_t current_device(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  return device_state(dev, out);
}

int pairs_for(int s_q, int H) { return (s_q * H + kRowsPerPair - 1) / kRowsPerPair; }

bool encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t row_bytes, uint32_t box_inner,
               uint32_t box_rows) {
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1_bytes,
               uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2) {
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1_bytes, s2_bytes};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool encode_kv_maps(PFN_cuTensorMapEncodeTiled_v12000 encode, KvMaps* maps, const void* kv_cache, int64_t num_blocks,
                    const void* q, int64_t q_rows) {
  const cuuint64_t strides[2] = {kDimQK * 2, 128};
  const cuuint32_t es[3] = {1, 1, 1};
  auto enc = [&](CUtensorMap* m, const void* base, int64_t rows, uint32_t chunk0_count) {
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), kDimQK / 64};
    const cuuint32_t box[3] = {64, 64, chunk0_count};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  const int64_t cache_rows = num_blocks * kPageTokens;
  // the sparse decode's row gathers: the cache as [row][576 dims], one 64-dim x 1-row box (a
  // tile::gather4 load reads four such rows)
  const cuuint64_t gdims[2] = {kDimQK, static_cast<cuuint64_t>(cache_rows)};
  const cuuint64_t gstrides[1] = {kDimQK * 2};
  const cuuint32_t gbox[2] = {64, 1};
  // (128-byte L2 fills: a gathered row is 1152 bytes, and 256-byte fills would overrun its end)
  const bool g4_ok = encode(&maps->g4, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(kv_cache), gdims,
                            gstrides, gbox, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  return g4_ok && enc(&maps->k_a, kv_cache, cache_rows, 5) && enc(&maps->c4, kv_cache, cache_rows, 4) &&
         enc(&maps->q, q, q_rows, kDimQK / 64);
}

bool encode_kv_maps_fp8(PFN_cuTensorMapEncodeTiled_v12000 encode, KvMaps* maps, const void* kv_cache,
                        int64_t num_blocks, const void* q, int64_t q_rows) {
  const cuuint64_t rows = static_cast<cuuint64_t>(num_blocks * kPageTokens);
  const cuuint32_t es[3] = {1, 1, 1};
  // the sparse decode's row gathers: the cache as [row][576 codes], one 128-code x 1-row box
  // (the RoPE chunk's box, at code 512, reads zeros past the row's end as the dense loads do).
  // 64-byte L2 fills: a 576-byte row starts 0 or 64 bytes into a 128-byte line, so 128-byte fills
  // would read 640 bytes a row.
  const cuuint64_t gdims[2] = {kDimQK, rows};
  const cuuint64_t gstrides[1] = {kDimQK};
  const cuuint32_t gbox[2] = {128, 1};
  const bool g4_ok = encode(&maps->g4, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(kv_cache), gdims,
                            gstrides, gbox, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_64B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  auto enc3 = [&](CUtensorMap* m, uint32_t chunks) {   // [chunk][row][128 codes] of dims 0..511
    const cuuint64_t dims[3] = {128, rows, kDimV / 128};
    const cuuint64_t strides[2] = {kDimQK, 128};
    const cuuint32_t box[3] = {128, 64, chunks};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(kv_cache), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  const cuuint64_t rdims[2] = {kDimQK, rows};
  const cuuint64_t rstrides[1] = {kDimQK};
  const cuuint32_t rbox[2] = {128, 64};
  const bool rope_ok = encode(&maps->rope, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(kv_cache), rdims,
                              rstrides, rbox, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  // q: bf16 [chunk 0..8][q row][64 dims] in boxes of 32 rows
  const cuuint64_t qdims[3] = {64, static_cast<cuuint64_t>(q_rows), kDimQK / 64};
  const cuuint64_t qstrides[2] = {kDimQK * 2, 128};
  const cuuint32_t qbox[3] = {64, 32, kDimQK / 64};
  const bool q_ok = encode(&maps->q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), qdims, qstrides, qbox,
                           es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  return g4_ok && enc3(&maps->k_a, 4) && enc3(&maps->c4, 2) && rope_ok && q_ok;
}

namespace {

size_t max_splits(int B, int num_parts) { return static_cast<size_t>(B) + static_cast<size_t>(num_parts); }

}  // namespace

int* device_status_word() {
  DeviceState* d = nullptr;
  if (current_device(&d) != MLA_OK) return nullptr;
  return d->status;
}

}  // namespace mla

using namespace mla;

extern "C" {

const char* mla_status_string(mla_status_t s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
    case MLA_ERR_DEVICE_BOUNDS: return "MLA_ERR_DEVICE_BOUNDS";
    default: return "MLA_ERR_UNKNOWN";
  }
}

int mla_num_sm_parts(int device, int s_q, int H) {
  if (s_q < 1 || H < 1) return -MLA_ERR_INVALID_ARG;
  const int n = pairs_for(s_q, H);
  if (n > kMaxPairsPerCluster) return -MLA_ERR_UNSUPPORTED;
  DeviceState* d = nullptr;
  const mla_status_t st = device_state(device, &d);
  if (st != MLA_OK) return -st;
  return d->parts[n];
}

size_t mla_metadata_size(int B, int num_sm_parts) {
  if (B < 0 || num_sm_parts < 1) return 0;
  return (static_cast<size_t>(kMetaInts) * num_sm_parts + B + 1) * sizeof(int32_t);
}

void mla_schedule_params(int* fixed_cost_pages, int* hbm_parts, int* split_cost_pages) {
  if (fixed_cost_pages) *fixed_cost_pages = kSegmentCostPages;
  if (hbm_parts) *hbm_parts = kHbmParts;
  if (split_cost_pages) *split_cost_pages = kSplitCostPages;
}

mla_status_t mla_decode_metadata(const int32_t* seqlens, int B, int s_q, int H, int causal_s_q, int num_sm_parts,
                                 void* metadata, mla_stream_t stream) {
  (void)causal_s_q;
  if (!seqlens || !metadata || B < 1 || s_q < 1 || H < 1 || num_sm_parts < 1) return MLA_ERR_INVALID_ARG;
  if (pairs_for(s_q, H) > kMaxPairsPerCluster || B > kScheduleMaxB) return MLA_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(metadata) & 3u) != 0) return MLA_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  mla_status_t st = current_device(&d);
  if (st != MLA_OK) return st;
  int32_t* meta = static_cast<int32_t*>(metadata);
  return launch_schedule(seqlens, B, num_sm_parts, kSegmentCostPages, kHbmParts, kSplitCostPages, meta, meta + kMetaInts * num_sm_parts,
                         reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

size_t mla_decode_workspace_size(int B, int s_q, int H, int num_sm_parts) {
  if (B < 1 || s_q < 1 || H < 1 || num_sm_parts < 1) return 0;
  const size_t rows = static_cast<size_t>(s_q) * H;
  const size_t ms = max_splits(B, num_sm_parts);
  const size_t o_bytes = ms * rows * kDimV * sizeof(float);
  const size_t l_bytes = ms * rows * sizeof(float);
  return o_bytes + ((l_bytes + 255) / 256) * 256;
}

}  // extern "C"

namespace {

// Shared body of mla_decode (indices == nullptr), mla_decode_sparse and mla_decode_fp8
// (kv_fp8: kv_cache holds E4M3 codes scaled by kv_scale).
mla_status_t decode_impl(const void* q, const void* kv_cache, int64_t num_blocks, const int32_t* block_table,
                         int max_blocks, const int32_t* seqlens, const int32_t* indices, int64_t idx_stride,
                         const int32_t* topk_lens, int B, int s_q, int H, float softmax_scale, int causal_s_q,
                         const void* metadata, int num_sm_parts, void* workspace, size_t workspace_bytes,
                         mla_bf16_t* out, float* lse, mla_stream_t stream, bool kv_fp8 = false,
                         float kv_scale = 1.f) {
  if (!q || !kv_cache || !block_table || !seqlens || !metadata || !out || !lse) return MLA_ERR_INVALID_ARG;
  if (B < 1 || s_q < 1 || H < 1 || num_blocks < 1 || max_blocks < 1 || num_sm_parts < 1) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(out) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seqlens) & 3u) ||
      (reinterpret_cast<uintptr_t>(metadata) & 3u))
    return MLA_ERR_INVALID_ARG;
  if (indices && (!topk_lens || idx_stride < 1 || (reinterpret_cast<uintptr_t>(indices) & 3u) ||
                  (reinterpret_cast<uintptr_t>(topk_lens) & 3u)))
    return MLA_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.f)) return MLA_ERR_INVALID_ARG;
  if (kv_fp8 && (!std::isfinite(kv_scale) || !(kv_scale > 0.f))) return MLA_ERR_INVALID_ARG;
  const int n_rb = pairs_for(s_q, H);
  if (n_rb > kMaxPairsPerCluster) return MLA_ERR_UNSUPPORTED;
  if (num_blocks * kPageTokens > (int64_t(1) << 31) - kPageTokens) return MLA_ERR_UNSUPPORTED;
  const size_t need = mla_decode_workspace_size(B, s_q, H, num_sm_parts);
  if (workspace_bytes < need || (need > 0 && !workspace)) return MLA_ERR_WORKSPACE;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return MLA_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  mla_status_t st = current_device(&d);
  if (st != MLA_OK) return st;

  KvMaps kv_maps;
  const int64_t q_rows = static_cast<int64_t>(B) * s_q * H;
  if (!(kv_fp8 ? encode_kv_maps_fp8(g_encode, &kv_maps, kv_cache, num_blocks, q, q_rows)
               : encode_kv_maps(g_encode, &kv_maps, kv_cache, num_blocks, q, q_rows)))
    return MLA_ERR_CUDA;

  const int rows = s_q * H;
  const size_t ms = max_splits(B, num_sm_parts);
  DecodeParams p;
  p.q = reinterpret_cast<const __nv_bfloat16*>(q);
  p.kv = reinterpret_cast<const __nv_bfloat16*>(kv_cache);
  p.num_blocks = num_blocks;
  p.block_table = block_table;
  p.max_blocks = max_blocks;
  p.seqlens = seqlens;
  p.lens = indices ? topk_lens : seqlens;
  p.indices = indices;
  p.idx_stride = indices ? idx_stride : 0;
  p.B = B;
  p.s_q = s_q;
  p.H = H;
  p.rows = rows;
  p.n_rb = n_rb;
  p.scale_log2 = static_cast<float>(static_cast<double>(softmax_scale) * 1.4426950408889634074);
  p.causal = causal_s_q ? 1 : 0;
  p.meta = static_cast<const int32_t*>(metadata);
  p.num_splits = p.meta + kMetaInts * num_sm_parts;
  p.num_parts = num_sm_parts;
  p.o_part = static_cast<float*>(workspace);
  p.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + ms * rows * kDimV * sizeof(float));
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.status = d->status;
  p.withhold_first_load = g_withhold_first_load;
  g_withhold_first_load = 0;
  p.kv_fp8 = kv_fp8 ? 1 : 0;
  p.kv_scale = kv_fp8 ? kv_scale : 1.f;

  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (launch_decode(kv_maps, p, 2 * n_rb, cs) != cudaSuccess) return MLA_ERR_CUDA;
  if (launch_combine(p.o_part, p.lse_part, p.num_splits, B, rows, static_cast<int>(ms), p.out, lse, p.status, cs) !=
      cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

}  // namespace

extern "C" {

mla_status_t mla_decode(const mla_bf16_t* q, const mla_bf16_t* kv_cache, int64_t num_blocks, const int32_t* block_table,
                        int max_blocks, const int32_t* seqlens, int B, int s_q, int H, float softmax_scale,
                        int causal_s_q, const void* metadata, int num_sm_parts, void* workspace,
                        size_t workspace_bytes, mla_bf16_t* out, float* lse, mla_stream_t stream) {
  return decode_impl(q, kv_cache, num_blocks, block_table, max_blocks, seqlens, nullptr, 0, nullptr, B, s_q, H,
                     softmax_scale, causal_s_q, metadata, num_sm_parts, workspace, workspace_bytes, out, lse, stream);
}

mla_status_t mla_decode_sparse(const mla_bf16_t* q, const mla_bf16_t* kv_cache, int64_t num_blocks,
                               const int32_t* block_table, int max_blocks, const int32_t* seqlens,
                               const int32_t* indices, int64_t index_stride, const int32_t* topk_lens, int B, int s_q,
                               int H, float softmax_scale, int causal_s_q, const void* metadata, int num_sm_parts,
                               void* workspace, size_t workspace_bytes, mla_bf16_t* out, float* lse,
                               mla_stream_t stream) {
  if (!indices) return MLA_ERR_INVALID_ARG;
  return decode_impl(q, kv_cache, num_blocks, block_table, max_blocks, seqlens, indices, index_stride, topk_lens, B,
                     s_q, H, softmax_scale, causal_s_q, metadata, num_sm_parts, workspace, workspace_bytes, out, lse,
                     stream);
}

mla_status_t mla_decode_sparse_fp8(const mla_bf16_t* q, const uint8_t* kv_cache, float kv_scale, int64_t num_blocks,
                                   const int32_t* block_table, int max_blocks, const int32_t* seqlens,
                                   const int32_t* indices, int64_t index_stride, const int32_t* topk_lens, int B,
                                   int s_q, int H, float softmax_scale, int causal_s_q, const void* metadata,
                                   int num_sm_parts, void* workspace, size_t workspace_bytes, mla_bf16_t* out,
                                   float* lse, mla_stream_t stream) {
  if (!indices) return MLA_ERR_INVALID_ARG;
  return decode_impl(q, kv_cache, num_blocks, block_table, max_blocks, seqlens, indices, index_stride, topk_lens, B,
                     s_q, H, softmax_scale, causal_s_q, metadata, num_sm_parts, workspace, workspace_bytes, out, lse,
                     stream, true, kv_scale);
}

mla_status_t mla_decode_fp8(const mla_bf16_t* q, const uint8_t* kv_cache, float kv_scale, int64_t num_blocks,
                            const int32_t* block_table, int max_blocks, const int32_t* seqlens, int B, int s_q, int H,
                            float softmax_scale, int causal_s_q, const void* metadata, int num_sm_parts,
                            void* workspace, size_t workspace_bytes, mla_bf16_t* out, float* lse,
                            mla_stream_t stream) {
  return decode_impl(q, kv_cache, num_blocks, block_table, max_blocks, seqlens, nullptr, 0, nullptr, B, s_q, H,
                     softmax_scale, causal_s_q, metadata, num_sm_parts, workspace, workspace_bytes, out, lse, stream,
                     true, kv_scale);
}

}  // extern "C"

namespace {

// Shared body of mla_absorb_q and mla_absorb_q_rope (positions == nullptr: plain copy of q_pe).
// With sched_meta set, one more CTA of the launch writes the split schedule of
// (sched_seqlens, sched_B, sched_parts) -- mla_decode_metadata's output -- to sched_meta.
mla_status_t absorb_impl(const mla_bf16_t* q_nope, int64_t q_nope_row_stride, const mla_bf16_t* q_pe,
                         int64_t q_pe_row_stride, const int32_t* positions, double rope_theta, const mla_bf16_t* w_uk,
                         mla_bf16_t* q, int N, int H, mla_stream_t stream, const int32_t* sched_seqlens = nullptr,
                         int sched_B = 0, int sched_parts = 0, int32_t* sched_meta = nullptr) {
  if (!q_nope || !w_uk || !q || N < 1 || H < 1) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_nope) || !aligned16(w_uk) || !aligned16(q)) return MLA_ERR_INVALID_ARG;
  if (q_nope_row_stride < static_cast<int64_t>(H) * 128 || (q_nope_row_stride % 8) != 0) return MLA_ERR_INVALID_ARG;
  if (q_pe && (!aligned16(q_pe) || q_pe_row_stride < static_cast<int64_t>(H) * 64 || (q_pe_row_stride % 8) != 0))
    return MLA_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  mla_status_t st = current_device(&d);
  if (st != MLA_OK) return st;
  CUtensorMap a_map, w_map;
  if (!encode_3d(&a_map, q_nope, 128, static_cast<uint64_t>(H), static_cast<uint64_t>(N), 256,
                 static_cast<uint64_t>(q_nope_row_stride) * 2, 64, 1, 128))
    return MLA_ERR_CUDA;
  if (!encode_2d(&w_map, w_uk, 512, static_cast<uint64_t>(H) * 128, 1024, 64, 64)) return MLA_ERR_CUDA;
  CUtensorMap o_map;   // q as [576, H, N], stored 64 columns x 32 rows at a time
  if (!encode_3d(&o_map, q, kDimQK, static_cast<uint64_t>(H), static_cast<uint64_t>(N), kDimQK * 2,
                 static_cast<uint64_t>(H) * kDimQK * 2, 64, 1, 32))
    return MLA_ERR_CUDA;
  BmmParams p = {};
  p.out = reinterpret_cast<__nv_bfloat16*>(q);
  p.out_row_stride = static_cast<int64_t>(H) * kDimQK;
  p.out_head_stride = kDimQK;
  p.N = N;
  p.H = H;
  p.status = d->status;
  p.pe = reinterpret_cast<const __nv_bfloat16*>(q_pe);
  p.pe_row_stride = q_pe_row_stride;
  p.positions = positions;
  p.w = reinterpret_cast<const __nv_bfloat16*>(w_uk);
  if (sched_meta) {
    p.sched_seqlens = sched_seqlens;
    p.sched_meta = sched_meta;
    p.sched_B = sched_B;
    p.sched_parts = sched_parts;
    p.sched_fixed = kSegmentCostPages;
    p.sched_hbm = kHbmParts;
    p.sched_split = kSplitCostPages;
  }
  if (positions) {   // inverse frequencies theta^(-2j/64) and 2*pi, each as a float pair (hi + lo)
    for (int j = 0; j < 32; ++j) {
      const double inv = std::pow(rope_theta, -2.0 * j / 64.0);
      p.rope_hi[j] = static_cast<float>(inv);
      p.rope_lo[j] = static_cast<float>(inv - static_cast<double>(p.rope_hi[j]));
    }
    const double two_pi = 6.283185307179586476925286766559;
    p.two_pi_hi = static_cast<float>(two_pi);
    p.two_pi_lo = static_cast<float>(two_pi - static_cast<double>(p.two_pi_hi));
  }
  return launch_bmm(true, a_map, w_map, o_map, p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

}  // namespace

extern "C" {

mla_status_t mla_absorb_q(const mla_bf16_t* q_nope, int64_t q_nope_row_stride, const mla_bf16_t* q_pe,
                          int64_t q_pe_row_stride, const mla_bf16_t* w_uk, mla_bf16_t* q, int N, int H,
                          mla_stream_t stream) {
  return absorb_impl(q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, nullptr, 0.0, w_uk, q, N, H, stream);
}

mla_status_t mla_absorb_q_rope(const mla_bf16_t* q_nope, int64_t q_nope_row_stride, const mla_bf16_t* q_pe,
                               int64_t q_pe_row_stride, const int32_t* positions, float rope_theta,
                               const mla_bf16_t* w_uk, mla_bf16_t* q, int N, int H, mla_stream_t stream) {
  if (!q_pe || !positions || (reinterpret_cast<uintptr_t>(positions) & 3u)) return MLA_ERR_INVALID_ARG;
  if (!std::isfinite(rope_theta) || !(rope_theta > 1.f)) return MLA_ERR_INVALID_ARG;
  return absorb_impl(q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, positions, static_cast<double>(rope_theta),
                     w_uk, q, N, H, stream);
}

int mla_absorb_plan_max_batch(void) { return kAbsorbPlanMaxB; }

mla_status_t mla_absorb_q_plan(const mla_bf16_t* q_nope, int64_t q_nope_row_stride, const mla_bf16_t* q_pe,
                               int64_t q_pe_row_stride, const int32_t* positions, float rope_theta,
                               const mla_bf16_t* w_uk, mla_bf16_t* q, int N, int H, const int32_t* seqlens, int B,
                               int num_sm_parts, void* metadata, mla_stream_t stream) {
  if (!seqlens || !metadata || B < 1 || num_sm_parts < 1 || N < 1 || H < 1 || N % B != 0) return MLA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(metadata) & 3u) != 0 || (reinterpret_cast<uintptr_t>(seqlens) & 3u) != 0)
    return MLA_ERR_INVALID_ARG;
  if (B > kAbsorbPlanMaxB || pairs_for(N / B, H) > kMaxPairsPerCluster) return MLA_ERR_UNSUPPORTED;
  if (positions) {
    if (!q_pe || (reinterpret_cast<uintptr_t>(positions) & 3u)) return MLA_ERR_INVALID_ARG;
    if (!std::isfinite(rope_theta) || !(rope_theta > 1.f)) return MLA_ERR_INVALID_ARG;
  }
  return absorb_impl(q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, positions, static_cast<double>(rope_theta),
                     w_uk, q, N, H, stream, seqlens, B, num_sm_parts, static_cast<int32_t*>(metadata));
}

mla_status_t mla_unabsorb_o(const mla_bf16_t* o_lat, const mla_bf16_t* w_uv, mla_bf16_t* o, int N, int H,
                            mla_stream_t stream) {
  if (!o_lat || !w_uv || !o || N < 1 || H < 1) return MLA_ERR_INVALID_ARG;
  if (!aligned16(o_lat) || !aligned16(w_uv) || !aligned16(o)) return MLA_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  mla_status_t st = current_device(&d);
  if (st != MLA_OK) return st;
  CUtensorMap a_map, w_map;
  if (!encode_3d(&a_map, o_lat, 512, static_cast<uint64_t>(H), static_cast<uint64_t>(N), 1024,
                 static_cast<uint64_t>(H) * 1024, 64, 1, 128))
    return MLA_ERR_CUDA;
  if (!encode_2d(&w_map, w_uv, 128, static_cast<uint64_t>(H) * 512, 256, 64, 64)) return MLA_ERR_CUDA;
  CUtensorMap o_map;   // o as [128, H, N], stored 64 columns x 32 rows at a time
  if (!encode_3d(&o_map, o, 128, static_cast<uint64_t>(H), static_cast<uint64_t>(N), 256,
                 static_cast<uint64_t>(H) * 256, 64, 1, 32))
    return MLA_ERR_CUDA;
  BmmParams p;
  p.out = reinterpret_cast<__nv_bfloat16*>(o);
  p.out_row_stride = static_cast<int64_t>(H) * 128;
  p.out_head_stride = 128;
  p.N = N;
  p.H = H;
  p.status = d->status;
  p.pe = nullptr;
  p.pe_row_stride = 0;
  p.positions = nullptr;
  p.w = reinterpret_cast<const __nv_bfloat16*>(w_uv);
  return launch_bmm(false, a_map, w_map, o_map, p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

size_t mla_bmm_fp8_workspace_size(void) { return static_cast<size_t>(kAmaxParts) * sizeof(float); }

}  // extern "C"

namespace {

// Shared body of mla_absorb_q_fp8 (absorb: x = q_nope, K = 128, 512 columns, optional q_pe
// copy / RoPE) and mla_unabsorb_o_fp8 (x = o_lat, K = 512, 128 columns).  With sched_meta
// set (absorb only), one more CTA of the amax launch writes the split schedule of
// (sched_seqlens, sched_B, sched_parts) to sched_meta.
mla_status_t bmm_fp8_impl(bool absorb, const mla_bf16_t* x, int64_t x_row_stride, const mla_bf16_t* q_pe,
                          int64_t q_pe_row_stride, const int32_t* positions, double rope_theta, const uint8_t* w_t,
                          float w_scale, mla_bf16_t* out, int N, int H, void* workspace, size_t workspace_bytes,
                          mla_stream_t stream, const int32_t* sched_seqlens = nullptr, int sched_B = 0,
                          int sched_parts = 0, int32_t* sched_meta = nullptr) {
  const int K = absorb ? 128 : kDimV;
  const int J = absorb ? kDimV : 128;
  if (!x || !w_t || !out || N < 1 || H < 1) return MLA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_t) || !aligned16(out)) return MLA_ERR_INVALID_ARG;
  if (x_row_stride < static_cast<int64_t>(H) * K || (x_row_stride % 8) != 0) return MLA_ERR_INVALID_ARG;
  if (q_pe && (!aligned16(q_pe) || q_pe_row_stride < static_cast<int64_t>(H) * 64 || (q_pe_row_stride % 8) != 0))
    return MLA_ERR_INVALID_ARG;
  if (!std::isfinite(w_scale) || !(w_scale > 0.f)) return MLA_ERR_INVALID_ARG;
  if (workspace_bytes < mla_bmm_fp8_workspace_size() || !workspace || (reinterpret_cast<uintptr_t>(workspace) & 15u))
    return workspace_bytes < mla_bmm_fp8_workspace_size() || !workspace ? MLA_ERR_WORKSPACE : MLA_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  mla_status_t st = current_device(&d);
  if (st != MLA_OK) return st;
  CUtensorMap x_map, w_map;
  // x as [K, H, N] with the token stride given: one box = 64 values of 128 tokens of one head
  if (!encode_3d(&x_map, x, static_cast<uint64_t>(K), static_cast<uint64_t>(H), static_cast<uint64_t>(N),
                 static_cast<uint64_t>(K) * 2, static_cast<uint64_t>(x_row_stride) * 2, 64, 1, 128))
    return MLA_ERR_CUDA;
  {   // the E4M3 weight codes as [H * J rows][K codes]: one box = 128 codes of the tile's rows
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(H) * J};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
    const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(absorb ? 256 : 128)};
    const cuuint32_t es[2] = {1, 1};
    if (g_encode(&w_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(w_t), dims, strides, box, es,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MLA_ERR_CUDA;
  }
  CUtensorMap o_map;   // out as [W, H, N] (W = 576 for q, 128 for o), stored 64 columns x 32 rows at a time
  {
    const uint64_t width = absorb ? kDimQK : 128;
    if (!encode_3d(&o_map, out, width, static_cast<uint64_t>(H), static_cast<uint64_t>(N), width * 2,
                   static_cast<uint64_t>(H) * width * 2, 64, 1, 32))
      return MLA_ERR_CUDA;
  }
  BmmFp8Params p = {};
  p.base.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.base.out_row_stride = static_cast<int64_t>(H) * (absorb ? kDimQK : 128);
  p.base.out_head_stride = absorb ? kDimQK : 128;
  p.base.N = N;
  p.base.H = H;
  p.base.status = d->status;
  p.base.pe = reinterpret_cast<const __nv_bfloat16*>(q_pe);
  p.base.pe_row_stride = q_pe_row_stride;
  p.base.positions = positions;
  if (positions) {   // inverse frequencies theta^(-2j/64) and 2*pi, each as a float pair (hi + lo)
    for (int j = 0; j < 32; ++j) {
      const double inv = std::pow(rope_theta, -2.0 * j / 64.0);
      p.base.rope_hi[j] = static_cast<float>(inv);
      p.base.rope_lo[j] = static_cast<float>(inv - static_cast<double>(p.base.rope_hi[j]));
    }
    const double two_pi = 6.283185307179586476925286766559;
    p.base.two_pi_hi = static_cast<float>(two_pi);
    p.base.two_pi_lo = static_cast<float>(two_pi - static_cast<double>(p.base.two_pi_hi));
  }
  if (sched_meta) {
    p.base.sched_seqlens = sched_seqlens;
    p.base.sched_meta = sched_meta;
    p.base.sched_B = sched_B;
    p.base.sched_parts = sched_parts;
    p.base.sched_fixed = kSegmentCostPages;
    p.base.sched_hbm = kHbmParts;
    p.base.sched_split = kSplitCostPages;
  }
  p.partials = static_cast<const float*>(workspace);
  p.w = w_t;
  p.J = J;
  p.w_scale = w_scale;
  return launch_bmm_fp8(absorb, reinterpret_cast<const __nv_bfloat16*>(x), x_row_stride, K, x_map, w_map, o_map, p,
                        static_cast<float*>(workspace), reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

}  // namespace

extern "C" {

mla_status_t mla_absorb_q_fp8(const mla_bf16_t* q_nope, int64_t q_nope_row_stride, const mla_bf16_t* q_pe,
                              int64_t q_pe_row_stride, const int32_t* positions, float rope_theta,
                              const uint8_t* w_uk_t, float w_uk_scale, mla_bf16_t* q, int N, int H, void* workspace,
                              size_t workspace_bytes, mla_stream_t stream) {
  if (positions && (!q_pe || (reinterpret_cast<uintptr_t>(positions) & 3u) || !std::isfinite(rope_theta) ||
                    !(rope_theta > 1.f)))
    return MLA_ERR_INVALID_ARG;
  return bmm_fp8_impl(true, q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, positions,
                      static_cast<double>(rope_theta), w_uk_t, w_uk_scale, q, N, H, workspace, workspace_bytes,
                      stream);
}

mla_status_t mla_absorb_q_fp8_plan(const mla_bf16_t* q_nope, int64_t q_nope_row_stride, const mla_bf16_t* q_pe,
                                   int64_t q_pe_row_stride, const int32_t* positions, float rope_theta,
                                   const uint8_t* w_uk_t, float w_uk_scale, mla_bf16_t* q, int N, int H,
                                   void* workspace, size_t workspace_bytes, const int32_t* seqlens, int B,
                                   int num_sm_parts, void* metadata, mla_stream_t stream) {
  if (!seqlens || !metadata || B < 1 || num_sm_parts < 1 || N < 1 || H < 1 || N % B != 0) return MLA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(metadata) & 3u) != 0 || (reinterpret_cast<uintptr_t>(seqlens) & 3u) != 0)
    return MLA_ERR_INVALID_ARG;
  if (B > kAbsorbPlanMaxB || pairs_for(N / B, H) > kMaxPairsPerCluster) return MLA_ERR_UNSUPPORTED;
  if (positions && (!q_pe || (reinterpret_cast<uintptr_t>(positions) & 3u) || !std::isfinite(rope_theta) ||
                    !(rope_theta > 1.f)))
    return MLA_ERR_INVALID_ARG;
  return bmm_fp8_impl(true, q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, positions,
                      static_cast<double>(rope_theta), w_uk_t, w_uk_scale, q, N, H, workspace, workspace_bytes,
                      stream, seqlens, B, num_sm_parts, static_cast<int32_t*>(metadata));
}

mla_status_t mla_unabsorb_o_fp8(const mla_bf16_t* o_lat, const uint8_t* w_uv_t, float w_uv_scale, mla_bf16_t* o, int N,
                                int H, void* workspace, size_t workspace_bytes, mla_stream_t stream) {
  if (!o_lat) return MLA_ERR_INVALID_ARG;
  return bmm_fp8_impl(false, o_lat, static_cast<int64_t>(H) * kDimV, nullptr, 0, nullptr, 0.0, w_uv_t, w_uv_scale, o, N,
                      H, workspace, workspace_bytes, stream);
}

namespace {
size_t round256(size_t x) { return (x + 255) / 256 * 256; }
int extend_cap(int chunk_tokens) { return (chunk_tokens + 127) / 128 * 128; }
}  // namespace

size_t mla_extend_workspace_size(int T, int H, int chunk_tokens) {
  if (T < 1 || H < 1 || chunk_tokens < kPageTokens || chunk_tokens % kPageTokens) return 0;
  const size_t cap = static_cast<size_t>(extend_cap(chunk_tokens));
  const size_t kv = round256(cap * H * 128 * sizeof(uint16_t));
  return 4 * kv + round256(static_cast<size_t>(T) * H * 128 * sizeof(float)) +
         round256(static_cast<size_t>(T) * H * sizeof(float));
}

mla_status_t mla_extend_chunked(const mla_bf16_t* q_nope, const mla_bf16_t* q_pe, const mla_bf16_t* w_uk,
                                const mla_bf16_t* w_uv, const mla_bf16_t* kv_cache, int64_t num_blocks,
                                const int32_t* block_row, int seqlen, int T, int H, float softmax_scale,
                                int chunk_tokens, void* workspace, size_t workspace_bytes, mla_bf16_t* out,
                                float* lse, mla_stream_t stream) {
  if (!q_nope || !q_pe || !w_uk || !w_uv || !kv_cache || !block_row || !out || !lse) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_nope) || !aligned16(q_pe) || !aligned16(w_uk) || !aligned16(w_uv) || !aligned16(kv_cache) ||
      !aligned16(out) || (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(block_row) & 3u))
    return MLA_ERR_INVALID_ARG;
  if (T < 1 || H < 1 || seqlen < T || num_blocks < 1) return MLA_ERR_INVALID_ARG;
  if (chunk_tokens < kPageTokens || chunk_tokens % kPageTokens) return MLA_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.f)) return MLA_ERR_INVALID_ARG;
  if (num_blocks * kPageTokens > (int64_t(1) << 31) - kPageTokens) return MLA_ERR_UNSUPPORTED;
  const size_t need = mla_extend_workspace_size(T, H, chunk_tokens);
  if (!workspace || workspace_bytes < need) return MLA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MLA_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  mla_status_t st = current_device(&d);
  if (st != MLA_OK) return st;

  const int cap = extend_cap(chunk_tokens);
  const uint64_t uH = static_cast<uint64_t>(H);
  ExtendMaps m;
  const bool maps_ok =
      encode_3d(&m.c, kv_cache, 64, static_cast<uint64_t>(num_blocks) * kPageTokens, kDimQK / 64, kDimQK * 2, 128, 64,
                64, 1) &&
      encode_2d(&m.wk, w_uk, kDimV, uH * 128, kDimV * 2, 64, 128) &&
      encode_2d(&m.wv, w_uv, 128, uH * kDimV, 256, 64, 64) &&
      encode_3d(&m.qn, q_nope, 128, uH, static_cast<uint64_t>(T), 256, uH * 256, 64, 1, 128) &&
      encode_3d(&m.qp, q_pe, 64, uH, static_cast<uint64_t>(T), 128, uH * 128, 64, 1, 128);
  char* ws = static_cast<char*>(workspace);
  const size_t kv_bytes = round256(static_cast<size_t>(cap) * H * 128 * sizeof(uint16_t));
  // two Kx / Vx buffers: chunk j expands into buffer j % 2, so that the expansion of chunk j + 1
  // may overlap the attention of chunk j
  __nv_bfloat16* kx[2] = {reinterpret_cast<__nv_bfloat16*>(ws), reinterpret_cast<__nv_bfloat16*>(ws + 2 * kv_bytes)};
  __nv_bfloat16* vx[2] = {reinterpret_cast<__nv_bfloat16*>(ws + kv_bytes),
                          reinterpret_cast<__nv_bfloat16*>(ws + 3 * kv_bytes)};
  float* acc_o = reinterpret_cast<float*>(ws + 4 * kv_bytes);
  float* acc_lse = reinterpret_cast<float*>(ws + 4 * kv_bytes + round256(static_cast<size_t>(T) * H * 128 * 4));
  // expanded keys and values head-major, [H][cap][128]: a 64-token tile of one head is 16 KiB in one run
  const uint64_t ucap = static_cast<uint64_t>(cap);
  if (!maps_ok) return MLA_ERR_CUDA;
  for (int i = 0; i < 2; ++i)
    if (!encode_3d(&m.kx[i], kx[i], 128, ucap, uH, 256, ucap * 256, 64, 64, 1) ||
        !encode_3d(&m.vx[i], vx[i], 128, ucap, uH, 256, ucap * 256, 64, 64, 1))
      return MLA_ERR_CUDA;
  m.kr = m.c;

  ExtendParams p;
  p.block_row = block_row;
  p.num_blocks = num_blocks;
  p.cap = cap;
  p.T = T;
  p.H = H;
  p.qpos0 = seqlen - T;
  p.scale_log2 = static_cast<float>(static_cast<double>(softmax_scale) * 1.4426950408889634074);

  p.acc_o = acc_o;
  p.acc_lse = acc_lse;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.status = d->status;
  const int n_chunks = (seqlen + chunk_tokens - 1) / chunk_tokens;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  for (int j = 0; j < n_chunks; ++j) {
    p.c0 = j * chunk_tokens;
    p.n = seqlen - p.c0 < chunk_tokens ? seqlen - p.c0 : chunk_tokens;
    p.first = j == 0;
    p.last = j == n_chunks - 1;
    p.defer_wait = j > 0;   // the first expansion may read cache rows the caller has just written
    p.kx = kx[j & 1];
    p.vx = vx[j & 1];
    if (launch_extend_chunk(m, p, j & 1, cs) != cudaSuccess) return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

mla_status_t mla_get_device_status(mla_stream_t stream) {
  DeviceState* d = nullptr;
  mla_status_t st = current_device(&d);
  if (st != MLA_OK) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return MLA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return MLA_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) return MLA_ERR_CUDA;
  return v;
}

void mla_debug_withhold_first_load(int enable) { g_withhold_first_load = enable ? 1 : 0; }

}  // extern "C"
