// mla_decode_noalloc: the decode path for callers that cannot allocate device memory.
//
// mla_decode asks the caller for two device buffers besides inputs and outputs:
// the tile-schedule metadata and the split workspace (fp32 partial outputs of
// requests whose KV range was split across SMs).  Some callers cannot provide
// them: code embedded in an inference engine or plugin whose memory pool hands
// out no scratch and whose fixed argument list has no slot for one, or a
// latency-critical decode loop that must never enter the allocator (cudaMalloc
// can synchronize the device and can fail under fragmentation).  This entry
// point needs only the inputs and outputs.  Its scratch lives in one fixed
// array in device memory, defined below, that every GPU loading this library
// holds until the process exits.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <cmath>
#include <mutex>

#include "mla_kernels.h"

namespace mla {
namespace {

// The scratch: schedule metadata in the first kMetaBytes, fp32 partials after it.
constexpr size_t kScratchBytes = size_t(64) << 20;     // 64 MiB per GPU
constexpr size_t kMetaBytes = size_t(256) << 10;       // room for 8*parts + B + 1 ints
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct NoallocDevice {
  bool ready = false;
  uint8_t* scratch = nullptr;   // device address of g_noalloc_scratch on this device
};
NoallocDevice g_na[kMaxDevices];
std::mutex g_na_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_na_encode = nullptr;

// Once per device, with that device current: resolve the scratch array's device
// address (in host code the array's name is only a host-side stand-in).
mla_status_t noalloc_setup(NoallocDevice** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_na_mutex);
  NoallocDevice& d = g_na[dev];
  if (!d.ready) {
    if (!g_na_encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return MLA_ERR_CUDA;
      g_na_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return MLA_ERR_CUDA;
    if (decode_set_attributes() != cudaSuccess) return MLA_ERR_CUDA;
    d.scratch = static_cast<uint8_t*>(ptr);
    d.ready = true;
  }
  *out = &d;
  return MLA_OK;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" mla_status_t mla_decode_noalloc(const mla_bf16_t* q, const mla_bf16_t* kv_cache, int64_t num_blocks,
                                           const int32_t* block_table, int max_blocks, const int32_t* seqlens,
                                           int B, int s_q, int H, float softmax_scale, int causal_s_q,
                                           int num_sm_parts, mla_bf16_t* out, float* lse, mla_stream_t stream) {
  if (!q || !kv_cache || !block_table || !seqlens || !out || !lse) return MLA_ERR_INVALID_ARG;
  if (B < 1 || s_q < 1 || H < 1 || num_blocks < 1 || max_blocks < 1 || num_sm_parts < 1) return MLA_ERR_INVALID_ARG;
  auto misaligned = [](const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0; };
  if (misaligned(q, 16) || misaligned(kv_cache, 16) || misaligned(out, 16) || misaligned(lse, 4) ||
      misaligned(block_table, 4) || misaligned(seqlens, 4))
    return MLA_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.f)) return MLA_ERR_INVALID_ARG;
  const int n_rb = (s_q * H + kRowsPerPair - 1) / kRowsPerPair;
  if (n_rb > kMaxPairsPerCluster || B > kScheduleMaxB) return MLA_ERR_UNSUPPORTED;
  if (num_blocks * kPageTokens > (int64_t(1) << 31) - kPageTokens) return MLA_ERR_UNSUPPORTED;
  // the sizes must fit the fixed scratch; larger problems are refused, not truncated
  const size_t meta_bytes = mla_metadata_size(B, num_sm_parts);
  const size_t ws_bytes = mla_decode_workspace_size(B, s_q, H, num_sm_parts);
  if (meta_bytes == 0 || meta_bytes > kMetaBytes || ws_bytes > kScratchBytes - kMetaBytes) return MLA_ERR_WORKSPACE;

  NoallocDevice* d = nullptr;
  mla_status_t st = noalloc_setup(&d);
  if (st != MLA_OK) return st;
  int* status = device_status_word();
  if (!status) return MLA_ERR_CUDA;

  KvMaps kv_maps;
  if (!encode_kv_maps(g_na_encode, &kv_maps, kv_cache, num_blocks, q, static_cast<int64_t>(B) * s_q * H))
    return MLA_ERR_CUDA;
  // Nothing in the scratch has to start at zero: the schedule kernel writes every
  // metadata entry, and the decode kernel writes each partial slot before the
  // combine kernel of the same call reads it.
  int32_t* meta = reinterpret_cast<int32_t*>(d->scratch);
  uint8_t* ws = d->scratch + kMetaBytes;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (launch_schedule(seqlens, B, num_sm_parts, kSegmentCostPages, kHbmParts, kSplitCostPages, meta, meta + kMetaInts * num_sm_parts,
                      cs) != cudaSuccess)
    return MLA_ERR_CUDA;

  const int rows = s_q * H;
  const size_t ms = static_cast<size_t>(B) + static_cast<size_t>(num_sm_parts);
  DecodeParams p;
  p.q = reinterpret_cast<const __nv_bfloat16*>(q);
  p.kv = reinterpret_cast<const __nv_bfloat16*>(kv_cache);
  p.num_blocks = num_blocks;
  p.block_table = block_table;
  p.max_blocks = max_blocks;
  p.seqlens = seqlens;
  p.lens = seqlens;
  p.indices = nullptr;
  p.idx_stride = 0;
  p.B = B;
  p.s_q = s_q;
  p.H = H;
  p.rows = rows;
  p.n_rb = n_rb;
  p.scale_log2 = static_cast<float>(static_cast<double>(softmax_scale) * 1.4426950408889634074);
  p.causal = causal_s_q ? 1 : 0;
  p.meta = meta;
  p.num_splits = meta + kMetaInts * num_sm_parts;
  p.num_parts = num_sm_parts;
  p.o_part = reinterpret_cast<float*>(ws);
  p.lse_part = reinterpret_cast<float*>(ws + ms * rows * kDimV * sizeof(float));
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.status = status;
  p.withhold_first_load = 0;
  if (launch_decode(kv_maps, p, 2 * n_rb, cs) != cudaSuccess) return MLA_ERR_CUDA;
  if (launch_combine(p.o_part, p.lse_part, p.num_splits, B, rows, static_cast<int>(ms), p.out, lse, p.status, cs) !=
      cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}
