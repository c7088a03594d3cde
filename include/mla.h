/*
 * mla.h -- C ABI of the GB300 (sm_103a) weight-absorbed MLA decode library.
 *
 * The operation (web page "MLA 推理：两条计算路径与 FlashMLA", section "两条等价的路径",
 * path 2; "DeepSeekV2之MLA", sections 4.3 and 4.5): with W_UK absorbed into the
 * query, decode attention is an MQA in which H query heads share one cached row
 * of 576 values per token -- the 512-dim latent c followed by the 64-dim shared
 * RoPE key k^R -- and the first 512 values are also the value vector.  For
 * request b, query position i (0 = earliest of the s_q new tokens), head h:
 *
 *     n     = seqlens[b]                       (no causal masking)
 *           = seqlens[b] - s_q + i + 1         (causal_s_q != 0)
 *     s_t   = softmax_scale * <q[b,i,h,0:576], kv_t[0:576]>,  t < n
 *     lse   = ln sum_t exp(s_t)                          (natural log, scaled scores)
 *     out   = sum_t exp(s_t - lse) * kv_t[0:512]
 *
 * with kv_t = kv_cache[block_table[b, t / 64], t % 64, :] (pages of 64 tokens, the
 * page size FlashMLA uses; same page, section "decode 注意力变成了计算问题").
 * A row with n = 0 gets out = 0 and lse = -inf.
 *
 * Conventions for every call:
 *  - Pointers are device pointers unless stated otherwise.  The caller allocates
 *    and owns every buffer (metadata and workspace included); the library never
 *    allocates or frees device memory.
 *  - bf16 = IEEE bfloat16 stored as uint16_t.  All tensors are dense, row-major,
 *    in the shapes given; q, kv_cache, out, q_nope, w_uk, w_uv, o_lat and o must
 *    be 16-byte aligned.
 *  - Every call is asynchronous on `stream` (0 = legacy default stream), except
 *    mla_get_device_status.  Argument errors are found on the host before any
 *    launch and returned as status codes; nothing aborts or throws.
 *  - Stream order holds as usual: every kernel sees the complete results of
 *    all work queued before it on the stream.  The kernels are launched with
 *    programmatic stream serialisation, so their launch and on-chip set-up may
 *    overlap the tail of the kernel queued just before them; they wait for that
 *    kernel to complete before their first global-memory access.  The calls
 *    may be recorded in CUDA graphs.
 *  - Device-side faults (a block-table entry outside [0, num_blocks), a barrier
 *    wait that ran out of time) do not trap: the kernels skip the access or end
 *    their loops and record a code in a device status word that
 *    mla_get_device_status reads.
 *  - Supported: 1 <= s_q * H <= 512 (rows are processed in blocks of 128;
 *    one block per 2-CTA pair, at most 4 pairs per cluster); 1 <= B <= 16384.
 *    Dims are fixed at 576 (q/k) and 512 (v); page size 64.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int mla_status_t;
#define MLA_OK                 0
#define MLA_ERR_INVALID_ARG    1   /* null/misaligned pointer, bad size           */
#define MLA_ERR_UNSUPPORTED    2   /* shape outside the supported set             */
#define MLA_ERR_WORKSPACE      3   /* metadata or workspace buffer too small      */
#define MLA_ERR_CUDA           4   /* a CUDA runtime/driver call failed           */
#define MLA_ERR_TIMEOUT        5   /* device: a bounded barrier wait ran out      */
#define MLA_ERR_DEVICE_BOUNDS  6   /* device: block-table entry out of range      */

typedef uint16_t mla_bf16_t;
typedef struct CUstream_st* mla_stream_t;   /* same handle as cudaStream_t */

/* Human-readable name of a status code (static string, never NULL). */
const char* mla_status_string(mla_status_t status);

/* Number of split parts (clusters of 2 * ceil(s_q*H/128) CTAs) that fit on the
 * device at once for this row count; the default num_sm_parts.  Returns <= 0 on
 * error (no device, unsupported rows). */
int mla_num_sm_parts(int device, int s_q, int H);

/* Bytes of the tile-schedule metadata for B requests and num_sm_parts parts. */
size_t mla_metadata_size(int B, int num_sm_parts);

/* Split-KV tile schedule ("get_mla_metadata": computed ahead of the kernel from
 * the sequence lengths only; page "MLA 推理：两条计算路径与 FlashMLA", FlashMLA
 * paragraph).  seqlens: [B] int32 device.  Writes metadata (mla_metadata_size
 * bytes, device): one 8-int record per part then B+1 split offsets.  The rule
 * (requests laid out in order on a line of cost positions -- a fixed set-up
 * cost per request, then one position per page -- cut into equal pieces, one
 * per part; hbm_parts parts are used when they already saturate the GPU's
 * bandwidth, all parts when that is estimated to pay for the extra splits) is
 * restated and checked bit for bit by the tests.  Reuse the
 * result for every layer of the same batch.  Async on stream. */
mla_status_t mla_decode_metadata(const int32_t* seqlens, int B, int s_q, int H, int causal_s_q,
                                 int num_sm_parts, void* metadata, mla_stream_t stream);

/* The schedule's constants, for tests: per-segment set-up cost (pages), the
 * number of parts that saturate HBM for one 2-CTA pair per part, and the cost of
 * an extra segment (pages) used to choose between that many parts and all of them.
 * Any pointer may be NULL. */
void mla_schedule_params(int* fixed_cost_pages, int* hbm_parts, int* split_cost_pages);

/* Bytes of the split workspace (fp32 partial outputs and lse of split requests). */
size_t mla_decode_workspace_size(int B, int s_q, int H, int num_sm_parts);

/* Absorbed MLA decode (see the header comment for the definition).
 *  q            [B, s_q, H, 576] bf16: [0:512) = q_nope.W_UK, [512:576) = RoPE'd q_pe
 *  kv_cache     [num_blocks, 64, 576] bf16 latent cache (16-byte aligned rows)
 *  block_table  [B, max_blocks] int32; only entries < ceil(seqlens[b]/64) are read
 *  seqlens      [B] int32, each in [0, max_blocks*64]; counts the s_q new tokens
 *  softmax_scale  finite and > 0 (else MLA_ERR_INVALID_ARG)
 *  metadata     from mla_decode_metadata with the same seqlens, B, s_q, H and
 *               num_sm_parts
 *  workspace    >= mla_decode_workspace_size bytes, 256-byte aligned
 *  out          [B, s_q, H, 512] bf16;  lse [B, s_q, H] fp32 (natural log)
 * Slots at or beyond seqlens[b] in the last page, and unused pages, may hold
 * anything (NaN included); they never reach the result.  Async on stream. */
mla_status_t mla_decode(const mla_bf16_t* q, const mla_bf16_t* kv_cache, int64_t num_blocks,
                        const int32_t* block_table, int max_blocks, const int32_t* seqlens,
                        int B, int s_q, int H, float softmax_scale, int causal_s_q,
                        const void* metadata, int num_sm_parts,
                        void* workspace, size_t workspace_bytes,
                        mla_bf16_t* out, float* lse, mla_stream_t stream);

/* Sparse (top-k) absorbed decode (web page "为什么 MLA + MTP 容易吃亏？从 Arithmetic
 * Intensity 看 Attention", section 6: a selector picks k of the cached latents --
 * DeepSeek-V3.2 keeps index_topk = 2048 -- and attention runs over those only, so
 * its cost follows k instead of the context length).  For request b, the list is
 * indices[b * index_stride + e], e < topk_lens[b]: token positions in [0, seqlens[b]),
 * looked up through the block table as in mla_decode.  Every query position and
 * head of the request attends to the listed tokens (with causal_s_q, query position
 * i drops listed tokens t > seqlens[b] - s_q + i):
 *     s_e = softmax_scale * <q[b,i,h,0:576], kv_t[0:576]>,  t = indices[b][e]
 *     lse = ln sum_e exp(s_e),   out = sum_e exp(s_e - lse) * kv_t[0:512]
 * A token listed twice counts twice.  An empty list gives out = 0, lse = -inf.
 *  indices      int32 device, 4-byte aligned; index_stride >= max topk_lens
 *  topk_lens    [B] int32 device, each in [0, index_stride]
 *  metadata     from mla_decode_metadata called with topk_lens in place of seqlens
 * Entries outside [0, seqlens[b]) are reported as MLA_ERR_DEVICE_BOUNDS (their rows
 * are skipped, the result is then undefined).  Other arguments as for mla_decode.
 * Async on stream. */
mla_status_t mla_decode_sparse(const mla_bf16_t* q, const mla_bf16_t* kv_cache, int64_t num_blocks,
                               const int32_t* block_table, int max_blocks, const int32_t* seqlens,
                               const int32_t* indices, int64_t index_stride, const int32_t* topk_lens, int B, int s_q,
                               int H, float softmax_scale, int causal_s_q, const void* metadata, int num_sm_parts,
                               void* workspace, size_t workspace_bytes, mla_bf16_t* out, float* lse,
                               mla_stream_t stream);

/* Absorbed decode over an FP8 latent cache (page "MLA 推理：两条计算路径与 FlashMLA":
 * the FlashMLA paragraph -- the kernel supports an FP8 KV cache -- and exercise 2 --
 * 576 bytes per cached token plus scale factors, which moves the decode from the
 * bandwidth limit to the tensor cores).
 *  kv_cache  [num_blocks, 64, 576] bytes: E4M3 codes (sign, 4 exponent bits with bias
 *            7, 3 mantissa bits; no infinities, codes 0x7F / 0xFF are NaN).  Cached
 *            value = code value * kv_scale.
 *  kv_scale  one scale for the whole cache, finite and > 0 (else MLA_ERR_INVALID_ARG)
 * The attention is that of mla_decode over the dequantized values; q stays bf16.
 * Inside, q (per row, scaled to the E4M3 range) and the probabilities are each carried
 * as a sum of two E4M3 terms for the FP8 tensor-core MMAs, which keeps the result
 * within the bf16 path's error.  Other arguments, results and errors as for mla_decode.
 * Async on stream. */
mla_status_t mla_decode_fp8(const mla_bf16_t* q, const uint8_t* kv_cache, float kv_scale, int64_t num_blocks,
                            const int32_t* block_table, int max_blocks, const int32_t* seqlens, int B, int s_q, int H,
                            float softmax_scale, int causal_s_q, const void* metadata, int num_sm_parts,
                            void* workspace, size_t workspace_bytes, mla_bf16_t* out, float* lse,
                            mla_stream_t stream);

/* The sparse (top-k) decode of mla_decode_sparse over an FP8 cache as in mla_decode_fp8:
 * the listed tokens' rows are E4M3 codes (576 bytes each) scaled by kv_scale.  Arguments,
 * results and errors as for those two calls.  Async on stream. */
mla_status_t mla_decode_sparse_fp8(const mla_bf16_t* q, const uint8_t* kv_cache, float kv_scale, int64_t num_blocks,
                                   const int32_t* block_table, int max_blocks, const int32_t* seqlens,
                                   const int32_t* indices, int64_t index_stride, const int32_t* topk_lens, int B,
                                   int s_q, int H, float softmax_scale, int causal_s_q, const void* metadata,
                                   int num_sm_parts, void* workspace, size_t workspace_bytes, mla_bf16_t* out,
                                   float* lse, mla_stream_t stream);

/* W_UK absorption and assembly of the decode query ("DeepSeekV2之MLA" 4.5:
 * q_nope_out = bmm(q_nope, w_kc) goes into q[..., :kv_lora_rank], the RoPE'd
 * q_pe into the last 64 values):
 *   q[n, h, 0:512]   = q_nope[n, h, 0:128] @ w_uk[h]    (fp32 accumulate, bf16 out)
 *   q[n, h, 512:576] = q_pe[n, h, 0:64]                 (copied; skipped if q_pe is NULL)
 *  q_nope  [N, H, 128] bf16, q_nope_row_stride elements between consecutive n
 *          (>= H*128, multiple of 8)
 *  q_pe    [N, H, 64] bf16 or NULL, q_pe_row_stride elements between consecutive n
 *          (>= H*64, multiple of 8)
 *  w_uk    [H, 128, 512] bf16
 *  q       [N, H, 576] bf16 (the decode q, N = B*s_q)
 * Async on stream.  The kernel is launched with programmatic stream serialization and
 * starts loading the weights before the previous kernel on the stream has finished (the
 * activations only after): the weights must not be written by the work queued just
 * before the call on the same stream (put an event or a synchronization in between if
 * they are).  The same holds for every absorption / un-absorption call below. */
mla_status_t mla_absorb_q(const mla_bf16_t* q_nope, int64_t q_nope_row_stride, const mla_bf16_t* q_pe,
                          int64_t q_pe_row_stride, const mla_bf16_t* w_uk, mla_bf16_t* q, int N, int H,
                          mla_stream_t stream);

/* mla_absorb_q with the RoPE of q_pe fused in (the query side of the decoupled
 * RoPE, page "MLA 推理：两条计算路径与 FlashMLA", section "两条等价的路径", its tiny
 * example: adjacent pairs rotated, written back interleaved):
 *   q[n, h, 512 + 2j]     = x0 cos(a) - x1 sin(a)
 *   q[n, h, 512 + 2j + 1] = x0 sin(a) + x1 cos(a),   x0, x1 = q_pe[n, h, 2j], q_pe[n, h, 2j+1]
 *   a = positions[n] * rope_theta^(-2j/64),  j = 0..31
 * (fp32 arithmetic on an angle reduced to within ~1e-7 rad, bf16 out).
 *  positions  [N] int32 device, each in [0, 2^24); 4-byte aligned
 *  rope_theta finite and > 1 (DeepSeek: 10000)
 * q_pe may not be NULL.  Other arguments as for mla_absorb_q.  Async on stream. */
mla_status_t mla_absorb_q_rope(const mla_bf16_t* q_nope, int64_t q_nope_row_stride, const mla_bf16_t* q_pe,
                               int64_t q_pe_row_stride, const int32_t* positions, float rope_theta,
                               const mla_bf16_t* w_uk, mla_bf16_t* q, int N, int H, mla_stream_t stream);

/* The W_UK absorption (mla_absorb_q_rope, or mla_absorb_q when positions is NULL)
 * and the split-KV schedule (mla_decode_metadata) in one launch: one CTA beyond the
 * absorption's tiles computes the schedule while the others multiply, so that the
 * decode issued next on the stream depends on a single kernel (its programmatic
 * launch then overlaps the absorption's tail instead of waiting on two).  Results
 * are those of the two separate calls, bit for bit.
 *  seqlens, B, num_sm_parts, metadata  as for mla_decode_metadata, with s_q = N / B
 *                                      (N a multiple of B) and the same H;
 *                                      B <= mla_absorb_plan_max_batch(), else
 *                                      MLA_ERR_UNSUPPORTED (the schedule's prefix sums
 *                                      live in that CTA's shared memory)
 *  the rest                            as for mla_absorb_q_rope (positions, rope_theta)
 *                                      or mla_absorb_q (positions NULL).
 * Async on stream. */
int mla_absorb_plan_max_batch(void);
mla_status_t mla_absorb_q_plan(const mla_bf16_t* q_nope, int64_t q_nope_row_stride, const mla_bf16_t* q_pe,
                               int64_t q_pe_row_stride, const int32_t* positions, float rope_theta,
                               const mla_bf16_t* w_uk, mla_bf16_t* q, int N, int H, const int32_t* seqlens, int B,
                               int num_sm_parts, void* metadata, mla_stream_t stream);

/* W_UV un-absorption ("DeepSeekV2之MLA" 4.5: bmm(attn_output, w_vc)):
 *   o[n, h, 0:128] = o_lat[n, h, 0:512] @ w_uv[h]      (fp32 accumulate, bf16 out)
 *  o_lat [N, H, 512] bf16 (the decode out), w_uv [H, 512, 128] bf16, o [N, H, 128] bf16.
 * Async on stream. */
mla_status_t mla_unabsorb_o(const mla_bf16_t* o_lat, const mla_bf16_t* w_uv, mla_bf16_t* o,
                            int N, int H, mla_stream_t stream);

/* FP8 projections (page "SGLang v0.3 MLA / torch.compile", the weight-absorption code
 * walk-through, its FP8 branches):  x_val, x_scale = input_to_float8(x);
 * y = bmm_fp8(x_val, w, x_scale, w_scale), one scale per operand, bf16 out.
 * The activation x is quantized per tensor inside the call: amax = max |x| over the whole
 * [N, H, K] tensor, inv = 448 / amax and x_scale = amax / 448 in float32 (1 and 1 when
 * amax = 0), codes = E4M3 round-to-nearest-even, saturating, of float32(x) * inv.  The
 * weights are E4M3 codes (sign, 4 exponent bits with bias 7, 3 mantissa bits) with one
 * per-tensor scale, each head's matrix stored transposed (K contiguous):
 *   y[n, h, j] = sum_k code_x[n, h, k] * code_w[h, j, k] * x_scale * w_scale
 * (fp32 accumulation on FP8 tensor cores, bf16 out).  A call runs two kernels on `stream`
 * (the maxima of |x|, then the product); `workspace` (device, 16-byte aligned, at least
 * mla_bmm_fp8_workspace_size() bytes, owned by the caller) carries the partial maxima
 * between them and may be reused by the next call on the same stream.  Too small or NULL:
 * MLA_ERR_WORKSPACE. */
size_t mla_bmm_fp8_workspace_size(void);

/* mla_absorb_q with FP8 weights (see above), K = 128:
 *   q[n, h, 0:512]   = bmm_fp8(input_to_float8(q_nope), W_UK)[n, h, :]
 *   q[n, h, 512:576] = q_pe[n, h, :], RoPE-rotated by positions[n] as in
 *                      mla_absorb_q_rope when positions is not NULL (copied when it is;
 *                      skipped when q_pe is NULL)
 *  w_uk_t      [H, 512, 128] E4M3 codes: W_UK[h] transposed;  w_uk_scale finite and > 0
 *  q_nope, q_pe, positions, rope_theta, q as for mla_absorb_q / mla_absorb_q_rope.
 * Async on stream. */
mla_status_t mla_absorb_q_fp8(const mla_bf16_t* q_nope, int64_t q_nope_row_stride, const mla_bf16_t* q_pe,
                              int64_t q_pe_row_stride, const int32_t* positions, float rope_theta,
                              const uint8_t* w_uk_t, float w_uk_scale, mla_bf16_t* q, int N, int H,
                              void* workspace, size_t workspace_bytes, mla_stream_t stream);

/* mla_absorb_q_fp8 and mla_decode_metadata in one pass: one CTA beyond the activation's
 * amax pass computes the split schedule, so that the decode issued next on the stream
 * depends on a single chain of kernels.  Results are those of the two separate calls,
 * bit for bit.  seqlens, B, num_sm_parts, metadata as for mla_absorb_q_plan (same limits);
 * the rest as for mla_absorb_q_fp8.  Async on stream. */
mla_status_t mla_absorb_q_fp8_plan(const mla_bf16_t* q_nope, int64_t q_nope_row_stride, const mla_bf16_t* q_pe,
                                   int64_t q_pe_row_stride, const int32_t* positions, float rope_theta,
                                   const uint8_t* w_uk_t, float w_uk_scale, mla_bf16_t* q, int N, int H,
                                   void* workspace, size_t workspace_bytes, const int32_t* seqlens, int B,
                                   int num_sm_parts, void* metadata, mla_stream_t stream);

/* mla_unabsorb_o with FP8 weights (see above), K = 512:
 *   o[n, h, 0:128] = bmm_fp8(input_to_float8(o_lat), W_UV)[n, h, :]
 *  o_lat [N, H, 512] bf16;  w_uv_t [H, 128, 512] E4M3 codes: W_UV[h] transposed;
 *  w_uv_scale finite and > 0;  o [N, H, 128] bf16.  Async on stream. */
mla_status_t mla_unabsorb_o_fp8(const mla_bf16_t* o_lat, const uint8_t* w_uv_t, float w_uv_scale, mla_bf16_t* o,
                                int N, int H, void* workspace, size_t workspace_bytes, mla_stream_t stream);

/* Chunked extend on the expanded path (MHA_CHUNKED_KV; page "MLA 推理：两条计算路径与
 * FlashMLA", end of section "两条等价的路径", and its exercise 3): T new tokens of one request
 * attend, causally, to the request's seqlen cached tokens, the new tokens being the last T
 * of them (new token i sits at position seqlen - T + i and sees positions <= its own).  The
 * cache is expanded chunk by chunk -- per head h and cached token t with latent c_t and RoPE
 * key k^R_t:  k_t = [W_UK[h] c_t (128), k^R_t (64)],  v_t = W_UV[h]^T c_t (128) -- each chunk
 * is attended to on its own, and the chunks' results are merged by log-sum-exp:
 *     s_t = softmax_scale * <[q_nope, q_pe][i, h], k_t>,   out = sum_t softmax(s)_t v_t,
 *     lse = ln sum_t exp(s_t)  (natural log, scaled scores)
 * so that the expanded context (~80 KB a token at H = 128) never exists at once.  The result
 * equals the absorbed path's (mla_absorb_q, then attention over the latent, then
 * mla_unabsorb_o) up to rounding.
 *  q_nope [T, H, 128], q_pe [T, H, 64] (RoPE applied) bf16;  w_uk [H, 128, 512] and
 *  w_uv [H, 512, 128] bf16 as for mla_absorb_q / mla_unabsorb_o;  kv_cache as for mla_decode;
 *  block_row: the request's block-table row, int32 device, entries for pages
 *  0 .. ceil(seqlen / 64) - 1 in [0, num_blocks) (others are reported as
 *  MLA_ERR_DEVICE_BOUNDS and read as zeros);  seqlen (host) >= T >= 1;
 *  chunk_tokens: cached tokens expanded at a time, a positive multiple of 64;
 *  workspace >= mla_extend_workspace_size(T, H, chunk_tokens) bytes, 256-byte aligned
 *  (two buffers of a chunk's expanded keys and values, ~512 * H bytes a chunk token each,
 *  so that the expansion of one chunk overlaps the attention of the chunk before, and the
 *  running fp32 merge of the output);  out [T, H, 128] bf16;  lse [T, H] fp32.
 * Launches two kernels per chunk on `stream`, in order (programmatic launches: the first
 * expansion waits for the work queued before the call, every later kernel for the one
 * before it, except that an expansion reads only the cache and the weights before the
 * previous chunk's attention has finished).  Async on stream. */
size_t mla_extend_workspace_size(int T, int H, int chunk_tokens);
mla_status_t mla_extend_chunked(const mla_bf16_t* q_nope, const mla_bf16_t* q_pe, const mla_bf16_t* w_uk,
                                const mla_bf16_t* w_uv, const mla_bf16_t* kv_cache, int64_t num_blocks,
                                const int32_t* block_row, int seqlen, int T, int H, float softmax_scale,
                                int chunk_tokens, void* workspace, size_t workspace_bytes, mla_bf16_t* out,
                                float* lse, mla_stream_t stream);

/* mla_decode without caller-provided scratch.  The paper has no counterpart:
 * this entry point exists for callers that cannot allocate device memory or pass
 * a workspace -- code inside an inference engine or plugin whose memory pool
 * hands out no scratch, or a decode loop that must never enter the allocator
 * (cudaMalloc can synchronize the device and fail under fragmentation).
 * It computes the split schedule and runs the same kernels as
 * mla_decode_metadata + mla_decode, with the schedule metadata and the fp32
 * split partials placed in one fixed 64 MiB array of device memory that the
 * library defines and that every GPU loading the library holds until exit.
 * Limits: mla_metadata_size(B, num_sm_parts) <= 256 KiB and
 * mla_decode_workspace_size(B, s_q, H, num_sm_parts) <= 64 MiB - 256 KiB, else
 * MLA_ERR_WORKSPACE and no launch (for H = 128, s_q = 1 that is
 * B + num_sm_parts <= 254).  It allocates nothing and calls no allocating routine.
 * The first call on a device resolves the array's device address (with that
 * device current); make that first call before any stream capture.  All calls
 * share the array and it keeps the last call's contents (nothing in it needs to
 * start at zero): calls whose kernels overlap on the GPU -- for example calls
 * on two streams of one process -- race on it and must be serialized by the
 * caller.  Arguments are those of mla_decode minus
 * metadata and workspace; the result is identical to mla_decode's for the same
 * num_sm_parts.  Async on stream. */
mla_status_t mla_decode_noalloc(const mla_bf16_t* q, const mla_bf16_t* kv_cache, int64_t num_blocks,
                                const int32_t* block_table, int max_blocks, const int32_t* seqlens,
                                int B, int s_q, int H, float softmax_scale, int causal_s_q, int num_sm_parts,
                                mla_bf16_t* out, float* lse, mla_stream_t stream);

/* Synchronizes `stream`, then reads and clears the device status word that the
 * kernels set (MLA_OK, MLA_ERR_TIMEOUT or MLA_ERR_DEVICE_BOUNDS). */
mla_status_t mla_get_device_status(mla_stream_t stream);

/* Test hook: when nonzero, the next mla_decode launch withholds the first KV
 * page load of every part, so that each barrier wait on it runs out of time
 * (0.5 s) and the call reports MLA_ERR_TIMEOUT through
 * mla_get_device_status.  No memory access is made out of bounds and nothing
 * traps; the flag clears itself after one launch. */
void mla_debug_withhold_first_load(int enable);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
