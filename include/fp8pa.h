/*
 * fp8pa.h -- C ABI of the GB300 (sm_103a) library for decode-step attention
 * over an FP8-quantised, paged KV cache.
 *
 * The method (as the source pages state it):
 *  - KV rows are stored as FP8 codes with an fp32 scale.  E4M3 has 4 exponent
 *    and 3 mantissa bits (range +-448, smallest non-zero 2^-9); E5M2 has 5 and
 *    2 (range +-57344) and is the format recommended for the KV cache for its
 *    range ("DeepSeek V4 950: whole-network FP8 dataflow",
 *    2kiu.com/news/4508674, sec. 2.1; "FP8混合精度推理全链路部署实战",
 *    ybb.press/ai-applications/14145.html, sec. 1.1 and sec. 2.2).
 *  - The scale of a group of values is absmax / 448 (absmax / 57344 for E5M2),
 *    clamped below at 1e-12, and the code is x / scale rounded to FP8
 *    ("Llama 3 70B FP8 deployment", dpshk.com/news/5605006, sec. 3.1).
 *  - The cache is paged: fixed-size blocks from one pool, one block table per
 *    request ("DeepSeek-V4.1 512K long-context TTFT", hotelren.com/news/5711065,
 *    sec. 3.3).
 *  - Attention is grouped-query (64 query heads share 8 KV heads for
 *    Llama-3-70B; dpshk.com/news/5605006 sec. 1.2) with the softmax in FP32
 *    (2kiu.com/news/4508674 sec. 2.3) computed as an online softmax
 *    (hotelren.com/news/5711065 sec. 2.2).
 *  - The MLA variant caches one compressed latent per token with one scale
 *    per latent group (2kiu.com/news/4508674 sec. 2.2).
 *
 * Conventions common to every call:
 *  - All data pointers are DEVICE pointers owned and allocated by the caller;
 *    the library allocates no memory (the decode's scratch is the caller's
 *    `workspace`).  bf16 arguments are raw bf16 bit patterns.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  The library never synchronises inside a call.
 *  - Return value: FP8PA_OK (0) or a negative FP8PA_ERR_* code.  When a call
 *    returns an error nothing was launched.
 *  - Bad indices found on the device (a slot or block id outside the pool, a
 *    sequence longer than its block table) never trap: the element is skipped
 *    and a bit is set in a per-device error word, read and cleared with
 *    fp8pa_get_device_error().
 *
 * Layouts (row-major, innermost last):
 *   codes            u8  [num_blocks][n_kv_heads][block_size][head_dim]
 *   TOKEN_HEAD scale f32 [num_blocks][n_kv_heads][block_size]
 *   TOKEN_GROUP scale f32 [num_blocks][n_kv_heads][block_size][head_dim/group_size]
 *   CHANNEL_STATIC scale f32 [n_kv_heads][head_dim]   (caller-given, read only)
 *   MX_BLOCK scale   u8  [num_blocks][n_kv_heads][block_size][head_dim/group_size]
 *                        (E8M0: byte b is the power of two 2^(b - 127); the
 *                        float* scale arguments then carry this byte buffer)
 *   SEGMENT scale    f32 [num_blocks][round_up(n_kv_heads, 4)]  (one 16-byte-
 *                        aligned row of page scales per block; the padding
 *                        entries are never read)
 *   slot s           -> block s / block_size, offset s % block_size
 *   block_tables     i32 [batch][max_blocks_per_seq]; token t of request b
 *                        lives in block block_tables[b][t / block_size]
 *   q                bf16 [batch][n_q_heads][head_dim]
 *   out              bf16 or f32 [batch][n_q_heads][head_dim_v]
 * Query head h reads KV head h / (n_q_heads / n_kv_heads).
 */
#ifndef FP8PA_H
#define FP8PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define FP8PA_OK 0
#define FP8PA_ERR_NULL_POINTER (-1)
#define FP8PA_ERR_BAD_ENUM (-2)
#define FP8PA_ERR_BAD_SHAPE (-3)
#define FP8PA_ERR_UNSUPPORTED (-4)
#define FP8PA_ERR_WORKSPACE (-5)
#define FP8PA_ERR_ALIGNMENT (-6)
#define FP8PA_ERR_CUDA (-7)

/* Bits of the device error word. */
#define FP8PA_DEVERR_SLOT_RANGE 1u   /* append: slot beyond num_blocks*block_size (row skipped) */
#define FP8PA_DEVERR_BLOCK_RANGE 2u  /* decode: block id outside [0, num_blocks) (page masked) */
#define FP8PA_DEVERR_SEQ_LEN 4u      /* decode: seq_len < 0 or > max_blocks_per_seq*block_size (clamped) */
#define FP8PA_DEVERR_TIMEOUT 8u      /* decode: a bounded wait on an async copy ran out (work abandoned) */

/* Code formats: FP8 E4M3 and E5M2, and symmetric INT8 (the alternate KV
 * codec; FMAX = 127, integer codes in [-127, 127] stored as the byte
 * integer + 128 (bytes 1 .. 255, 128 for zero), value = byte - 128; not
 * with FP8PA_SCALE_MX_BLOCK). */
#define FP8PA_E4M3 0
#define FP8PA_E5M2 1
#define FP8PA_INT8 2

/* Scale granularities. */
#define FP8PA_SCALE_TOKEN_HEAD 0     /* dynamic: one f32 per (token, kv head), written by append */
#define FP8PA_SCALE_CHANNEL_STATIC 1 /* static: caller-given f32 per (kv head, dim), read only   */
#define FP8PA_SCALE_TOKEN_GROUP 2    /* dynamic: one f32 per (token, kv head, group of dims)     */
#define FP8PA_SCALE_MX_BLOCK 3       /* dynamic: one E8M0 byte per (token, kv head, 16/32 dims)  */
#define FP8PA_SCALE_SEGMENT 4        /* cumulative: one f32 per (page, kv head), 1024-token segments */

/* Tokens per segment of FP8PA_SCALE_SEGMENT. */
#define FP8PA_SEGMENT_TOKENS 1024

/* Output element types of the decode. */
#define FP8PA_OUT_BF16 0
#define FP8PA_OUT_F32 1

/*
 * Append new tokens' K/V rows to the cache.
 * Defined by: absmax scale and FP8 cast, "Llama 3 70B FP8 deployment"
 * (dpshk.com/news/5605006) sec. 3.1; per-latent-group scales,
 * "DeepSeek V4 950" (2kiu.com/news/4508674) sec. 2.2; paged blocks,
 * "DeepSeek-V4.1 512K" (hotelren.com/news/5711065) sec. 3.3.
 *
 * k, v          bf16 [num_tokens][n_kv_heads][head_dim]; v may be NULL (then
 *               v_cache/v_scale are ignored: the single-latent MLA cache).
 * slot_mapping  i32 [num_tokens]; a negative slot skips that token.  Two
 *               tokens with the same slot in one call race (undefined).
 * fmt           FP8PA_E4M3, FP8PA_E5M2 or FP8PA_INT8 (FMAX 127 in every
 *               scale below).
 * scale_mode    TOKEN_HEAD: s = max(absmax(row)/FMAX, 1e-12), written to
 *               k_scale/v_scale.  TOKEN_GROUP: the same per group of
 *               group_size dims.  CHANNEL_STATIC: s = k_scale[h][d] given
 *               by the caller, not written.  MX_BLOCK: per block of
 *               group_size (16 or 32) dims the power of two s = 2^e,
 *               e = floor(log2(absmax)) - emax (emax 8 for E4M3, 15 for
 *               E5M2) held in [-127, 127] (-127 for an all-zero block),
 *               written as the byte e + 127 -- the Microscaling block format
 *               that "FP8混合精度推理全链路部署实战"
 *               (ybb.press/ai-applications/14145.html) sec. 7.1 names for
 *               Blackwell; codes = fp8_rne_satfinite(x * 2^-e), exact scaling.
 * code          = fp8_rne_satfinite(x / s), IEEE fp32 division; INT8:
 *               x / s rounded to the nearest integer, ties to even, clamped
 *               to [-127, 127], stored + 128 (an INT8 KV cache is named only as a serving
 *               option, hotelren.com/news/5166672, inference-engine settings;
 *               the rest is this library's reading).  Codes are bit-exact
 *               with the definition above.  MX_BLOCK is FP8 only
 *               (FP8PA_ERR_UNSUPPORTED with INT8).
 * Requirements  head_dim % 16 == 0, head_dim <= 768; group_size in
 *               {16,32,64,128,256} dividing head_dim ({16,32} for MX_BLOCK);
 *               block_size > 0;
 *               16-byte aligned k, v, caches and scales.
 * Errors        negative code, nothing launched.  A slot past the pool is
 *               skipped and sets FP8PA_DEVERR_SLOT_RANGE.
 */
int fp8pa_kv_append_quant(const void* k, const void* v, const int32_t* slot_mapping,
                          int num_tokens, int n_kv_heads, int head_dim, int fmt, int scale_mode,
                          int group_size, uint8_t* k_cache, uint8_t* v_cache, float* k_scale,
                          float* v_scale, int num_blocks, int block_size, void* stream);

/*
 * Append with block-wise cumulative rescaling (FP8PA_SCALE_SEGMENT).
 * Defined by: "DeepSeek V4 950: whole-network FP8 dataflow"
 * (2kiu.com/news/4508674) sec. 4.3 -- the KV cache is cut into length
 * blocks, each keeps a cumulative scale that decode re-aligns by, and an
 * extra offset beyond the per-head scale is refreshed every 1024 tokens.
 * The page gives no formula; this library's reading:
 *   per (sequence, K or V, kv head) a running absmax R covers every token
 *   appended so far (restarting at position 0).  Appending the token at
 *   position p sets R = max(R, absmax(row)); if p is a multiple of
 *   FP8PA_SEGMENT_TOKENS the token opens a segment and its scale is frozen
 *   as S = max(R / FMAX, 1e-12) (IEEE fp32 division).  Every token of the
 *   segment is coded as fp8_rne_satfinite(x / S) (INT8: as in
 *   fp8pa_kv_append_quant) and each page stores S once per kv head.
 *   A value beyond S * FMAX inside a segment saturates; the next segment's
 *   scale covers it.
 *
 * k, v           bf16 [num_tokens][n_kv_heads][head_dim]; v may be NULL.
 * seq_offsets    i32 [num_seqs + 1] (device): sequence r owns rows
 *                seq_offsets[r] .. seq_offsets[r+1]-1, in position order.
 * seq_start_pos  i32 [num_seqs] (device): position of sequence r's first
 *                row in this call (its cached length before the call).
 * slot_mapping   i32 [num_tokens]; a negative slot, or one past the pool
 *                (flagged FP8PA_DEVERR_SLOT_RANGE), skips the token: it
 *                neither raises R nor opens its segment.
 * seg_state      f32 [num_seqs][2][n_kv_heads][2] (device, caller-owned):
 *                (R, S) of each (sequence, K or V, head), carried between
 *                calls; row r belongs to the call's sequence r, so a caller
 *                that reorders its batch reorders these rows with it.  Rows
 *                of a sequence starting at position 0 need no initialisation.
 * k_scale, v_scale  f32 [num_blocks][round_up(n_kv_heads, 4)]: written.
 * Requirements   block_size divides FP8PA_SEGMENT_TOKENS; head_dim % 16 == 0,
 *                head_dim <= 768; 16-byte aligned k, v, caches and scales.
 * Codes and scales are bit-exact with the definition above, whatever the
 * split of a sequence's tokens into calls.  Decode reads the page scales
 * with scale_mode FP8PA_SCALE_SEGMENT.  Calls that touch the same sequence
 * must be stream-ordered.
 */
int fp8pa_kv_append_quant_segment(const void* k, const void* v, const int32_t* slot_mapping,
                                  const int32_t* seq_offsets, const int32_t* seq_start_pos,
                                  int num_seqs, int n_kv_heads, int head_dim, int fmt,
                                  float* seg_state, uint8_t* k_cache, uint8_t* v_cache,
                                  float* k_scale, float* v_scale, int num_blocks, int block_size,
                                  void* stream);

/*
 * Static per-channel scales for CHANNEL_STATIC mode: for every (kv head, dim)
 * s = max(absmax over the num_tokens rows / FMAX, 1e-12).
 * Defined by: per-channel KV scales, "DeepSeek-V4.1 512K"
 * (hotelren.com/news/5711065) sec. 3.3; absmax / FMAX, dpshk.com/news/5605006
 * sec. 3.1.
 * x          bf16 [num_tokens][n_kv_heads][head_dim].
 * scale_out  f32 [n_kv_heads][head_dim], overwritten (used as scratch for the
 *            running maximum during the call).
 */
int fp8pa_kv_channel_scales(const void* x, int num_tokens, int n_kv_heads, int head_dim, int fmt,
                            float* scale_out, void* stream);

/*
 * Online calibration of static per-channel scales, one prefill batch at a
 * time: running_absmax[h][d] = max(running_absmax[h][d], max_t |x[t][h][d]|).
 * Defined by: a running maximum per attention layer, updated with each
 * prefill batch and used for the scales of later tokens, after a warm-up on
 * representative inputs ("Llama 3 70B FP8 deployment", dpshk.com/news/5605006,
 * sec. 3.2).
 * x               bf16 [num_tokens][n_kv_heads][head_dim].
 * running_absmax  f32 [n_kv_heads][head_dim], caller-owned, zero before the
 *                 first batch, updated in place (values stay non-negative).
 * Calls on the same running_absmax are commutative (order does not matter).
 */
int fp8pa_kv_channel_absmax_update(const void* x, int num_tokens, int n_kv_heads, int head_dim,
                                   float* running_absmax, void* stream);

/*
 * Static scales from a running absmax: scale[i] = max(absmax[i] / FMAX, 1e-12)
 * (IEEE fp32 division; dpshk.com/news/5605006 sec. 3.1).  n = n_kv_heads *
 * head_dim.  scale_out may alias absmax.
 */
int fp8pa_kv_scales_from_absmax(const float* absmax, int n, int fmt, float* scale_out,
                                void* stream);

/*
 * Bytes of device workspace fp8pa_paged_decode_attention needs for these
 * shapes on the current device (it depends on the device's SM count); enough
 * for every scale mode and format.  0 if the shapes are rejected.
 */
size_t fp8pa_decode_workspace_bytes(int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                    int head_dim_v, int block_size, int max_blocks_per_seq);

/*
 * The same for fp8pa_paged_multiquery_attention (and fp8pa_decode_step) with
 * q_len queries per request; q_len = 1 is fp8pa_decode_workspace_bytes.
 */
size_t fp8pa_multiquery_workspace_bytes(int batch, int q_len, int n_q_heads, int n_kv_heads,
                                        int head_dim, int head_dim_v, int block_size,
                                        int max_blocks_per_seq);

/*
 * Decode-step attention of one query token per request over its paged,
 * FP8-quantised cache: out[b][h] = sum_t softmax_t(sm_scale * q[b][h] . k^_t)
 * * v^_t over t < seq_lens[b], with k^ = decode(code) * scale.
 * Defined by: GQA, dpshk.com/news/5605006 sec. 1.2; FP32 softmax,
 * 2kiu.com/news/4508674 sec. 2.3; blockwise online softmax,
 * hotelren.com/news/5711065 sec. 2.2; paged blocks, same page sec. 3.3;
 * MLA latent, 2kiu.com/news/4508674 sec. 2.2.
 *
 * Long contexts are split into chunks across the whole GPU and the per-chunk
 * partials (running max, sum, unnormalised output) are merged by a second
 * pass; the result does not depend on the split beyond fp32 rounding.
 *
 * Two layouts are served:
 *  GQA  n_q_heads % n_kv_heads == 0, n_q_heads/n_kv_heads <= 8, head_dim in
 *       {64, 128}, head_dim_v == head_dim, block_size in {16, 32, 64},
 *       scale_mode TOKEN_HEAD, CHANNEL_STATIC, MX_BLOCK (group_size 16
 *       or 32, FP8 codes) or SEGMENT, separate v_cache/v_scale.
 *  MLA  n_kv_heads == 1, head_dim 576 (512 latent + 64 rope), head_dim_v
 *       512 (the first 512 dims of the same latent), v_cache == k_cache,
 *       v_scale == k_scale, scale_mode TOKEN_GROUP (group_size 64) or
 *       SEGMENT, block_size 64, n_q_heads a multiple of 32.
 *
 * fmt          FP8PA_E4M3, FP8PA_E5M2 or FP8PA_INT8: the codes as
 *              fp8pa_kv_append_quant wrote them (decoded exactly to f16).
 * seq_lens     i32 [batch], including any token appended this step; 0 gives
 *              a zero output row.
 * num_blocks   size of the pool (bounds block ids; sizes the copy maps).
 * out_dtype    FP8PA_OUT_BF16 (round to nearest even) or FP8PA_OUT_F32.
 * workspace    device scratch of at least fp8pa_decode_workspace_bytes();
 *              16-byte aligned; contents need no initialisation.  Calls that
 *              share a workspace must be stream-ordered.
 * Errors       negative code, nothing launched.  Bad block ids or lengths
 *              are masked on the device and set an error bit.
 */
int fp8pa_paged_decode_attention(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                 const float* k_scale, const float* v_scale,
                                 const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* seq_lens, int batch, int block_size,
                                 int n_q_heads, int n_kv_heads, int head_dim, int head_dim_v,
                                 int fmt, int scale_mode, int group_size, float sm_scale,
                                 int num_blocks, void* out, int out_dtype, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * Attention of a causal chunk of q_len query tokens per request over the
 * paged FP8 cache: the chunk's own tokens were appended to the cache first,
 * so query i (0 <= i < q_len) of request b sees the first
 * seq_lens[b] - (q_len - 1 - i) cached tokens, and the last query sees them
 * all.  q_len = 1 is fp8pa_paged_decode_attention.
 * Serves the chunks that a scheduler interleaves with decode steps when it
 * splits a long prompt (chunked prefill: dpshk.com/news/5605006, sec. 2.1 and
 * 3.3; hotelren.com/news/5711065, sec. 3.4) and the verify step of
 * speculative decoding, where the target model scores several draft tokens
 * at once (dpshk.com/news/5605006, sec. 4.3).  Each query row is computed
 * exactly as a decode row over its visible prefix.
 *
 * q            bf16 [batch][q_len][n_q_heads][head_dim].
 * out          [batch][q_len][n_q_heads][head_dim_v], bf16 or f32.
 *              Chunks of q_len 2..8 on the GQA layout with E4M3/E5M2 codes,
 *              TOKEN_HEAD scales, head_dim 128 and G = n_q_heads/n_kv_heads
 *              such that G x qw is 16 or 32 for some qw dividing q_len run
 *              on the tensor cores, qw queries at a time; those also accept
 *              G up to 32.
 * seq_lens     i32 [batch], the cached length including the whole chunk.
 *              A request shorter than q_len (or outside [0, cap]) sets
 *              FP8PA_DEVERR_SEQ_LEN; its rows that would see no token are 0.
 * workspace    at least fp8pa_multiquery_workspace_bytes(batch, q_len, ...).
 * Layout limits, other arguments and errors as fp8pa_paged_decode_attention;
 * q_len <= 0 returns FP8PA_ERR_BAD_SHAPE.
 */
int fp8pa_paged_multiquery_attention(const void* q, const uint8_t* k_cache,
                                     const uint8_t* v_cache, const float* k_scale,
                                     const float* v_scale, const int32_t* block_tables,
                                     int max_blocks_per_seq, const int32_t* seq_lens, int batch,
                                     int q_len, int block_size, int n_q_heads, int n_kv_heads,
                                     int head_dim, int head_dim_v, int fmt, int scale_mode,
                                     int group_size, float sm_scale, int num_blocks, void* out,
                                     int out_dtype, void* workspace, size_t workspace_bytes,
                                     void* stream);

/*
 * One decode step in one call: the append of fp8pa_kv_append_quant
 * (k_new, v_new, slot_mapping, num_new_tokens into the cache), then the
 * attention of fp8pa_paged_multiquery_attention over the updated cache
 * (q_len = 1: fp8pa_paged_decode_attention).  The result equals the two
 * calls made in that order, bit for bit; the split planner runs inside the
 * append's launch, so the step is three kernel launches instead of four.
 * Defined by: the two steps of the decode path, append then attend
 * ("Llama 3 70B FP8 deployment", dpshk.com/news/5605006, sec. 3.2: decode
 * quantises each new KV with the current scale; "DeepSeek-V4.1 512K",
 * hotelren.com/news/5711065, sec. 3.3: paged KV blocks).
 * Arguments, layouts, errors: those of the two calls; the cache and scale
 * tensors are shared by both.  Nothing is launched if either argument set
 * is rejected.  FP8PA_SCALE_SEGMENT is not served here (its append needs
 * token positions: call fp8pa_kv_append_quant_segment, then the attention).
 */
int fp8pa_decode_step(const void* k_new, const void* v_new, const int32_t* slot_mapping,
                      int num_new_tokens, const void* q, uint8_t* k_cache, uint8_t* v_cache,
                      float* k_scale, float* v_scale, const int32_t* block_tables,
                      int max_blocks_per_seq, const int32_t* seq_lens, int batch, int q_len,
                      int block_size, int n_q_heads, int n_kv_heads, int head_dim,
                      int head_dim_v, int fmt, int scale_mode, int group_size, float sm_scale,
                      int num_blocks, void* out, int out_dtype, void* workspace,
                      size_t workspace_bytes, void* stream);

/*
 * Size of the scratch array built into the library for
 * fp8pa_paged_decode_attention_static_ws.  The array is reserved on a device
 * when the library's module is loaded there: on its first use under lazy
 * module loading (the CUDA default), at context creation under
 * CUDA_MODULE_LOADING=EAGER, whether or not this call is ever made.  It is
 * held until the process exits (or the device is reset).
 */
#define FP8PA_STATIC_WORKSPACE_BYTES (32u << 20)

/*
 * The source pages have no counterpart to this call; it serves users of the
 * library who cannot allocate device memory -- for example a plugin whose
 * host framework passes it only the input and output buffers and owns the
 * allocator, or a server that fixes its memory at start-up and allows no
 * allocation afterwards.
 *
 * Same arguments and result as fp8pa_paged_decode_attention, minus the
 * workspace: the scratch comes from a static device array of
 * FP8PA_STATIC_WORKSPACE_BYTES inside the library, so the call allocates
 * nothing (no cudaMalloc, no allocator of any library).  The caller still
 * owns every input and the output.
 *  - Every call made outside stream capture looks the array's device address
 *    up again (with the calling device current), so a device reset between
 *    calls is safe.  A call made during a capture reuses the address the
 *    last uncaptured call on that device found: make the first call on each
 *    device before any stream capture.
 *  - Every call on a device shares the one array; calls whose kernels may
 *    overlap on the GPU (unordered streams) race and give undefined output.
 *    Nothing in the array needs clearing between calls.
 *  - A call whose own workspace need (for its shapes, format, scale mode and
 *    split; at most fp8pa_decode_workspace_bytes) exceeds
 *    FP8PA_STATIC_WORKSPACE_BYTES returns FP8PA_ERR_WORKSPACE and launches
 *    nothing; other errors are those of fp8pa_paged_decode_attention.
 */
int fp8pa_paged_decode_attention_static_ws(const void* q, const uint8_t* k_cache,
                                           const uint8_t* v_cache, const float* k_scale,
                                           const float* v_scale, const int32_t* block_tables,
                                           int max_blocks_per_seq, const int32_t* seq_lens,
                                           int batch, int block_size, int n_q_heads,
                                           int n_kv_heads, int head_dim, int head_dim_v, int fmt,
                                           int scale_mode, int group_size, float sm_scale,
                                           int num_blocks, void* out, int out_dtype,
                                           void* stream);

/*
 * Synchronise `stream`, then return (in *flags) and clear the current
 * device's error word.  Returns FP8PA_OK or FP8PA_ERR_CUDA.
 */
int fp8pa_get_device_error(void* stream, uint32_t* flags);

/*
 * Self-test of the bounded waits every kernel uses on its asynchronous
 * copies: one warp waits on a shared-memory barrier that nothing completes,
 * for at most `limit_cycles` SM cycles (clamped to [1e3, 4e9]), then records
 * FP8PA_DEVERR_TIMEOUT in the device error word and returns -- exactly what
 * a decode warp does when a copy never lands.  Read the result with
 * fp8pa_get_device_error().  Nothing is faulted, trapped or left hanging.
 */
int fp8pa_selftest_bounded_wait(long long limit_cycles, void* stream);

/*
 * TESTING AND BENCHMARKING ONLY -- not for production callers.
 * The two calls below set process-global state that every later decode call
 * of every thread reads, with no synchronisation: they are not thread-safe,
 * and a change made while another thread is inside a decode call, or while
 * a decode call is being captured into a CUDA graph, has undefined effect.
 * Set them only while no other thread uses the library.
 */

/*
 * Test hook: the number of split workers the decode uses (0 = one per
 * resident warp slot on the device, the default).  It changes how the
 * sequences are cut into partials, never the result beyond fp32 rounding;
 * the tests use it to run every kind of page range.  It also changes
 * fp8pa_decode_workspace_bytes().
 */
int fp8pa_set_decode_workers(int workers);

/*
 * Measurement hook: when both events are non-NULL (cudaEvent_t handles),
 * every later decode call records `start` on its stream immediately before
 * its split kernel and `stop` immediately after it, so a benchmark can time
 * the dominant kernel alone.  NULL, NULL turns it off.
 */
int fp8pa_set_split_events(void* start, void* stop);

/* Static text for a status code. */
const char* fp8pa_error_string(int code);

/* ABI version: (major << 16) | minor. */
int fp8pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8PA_H */
