/*
 * gqa_attn.h — C ABI of the GB300 (sm_103a) grouped-query softmax attention
 * forward library, libgqa_attn.so.
 *
 * Operation (TileOPs "Attention Operators", GQADenseFwdOp, stages 1-7, and
 * RL-Kernel "Standard Softmax Attention", Accuracy):
 *
 *     O[b,i,h,:] = sum_{j in V(b,i)} softmax_j( scale * <q[b,i,h,:], k[b,j,r,:]> ) * v[b,j,r,:]
 *
 *   r = h / (Hq / Hkv)                     query head h reads KV head r
 *   p_i = i + Skv - Sq                     queries aligned to the end of the keys
 *   V(b,i) = { j < Skv : (!causal || j <= p_i) && key_padding_mask[b,j] != 0 }
 *
 * Accumulation is FP32; O is written as bfloat16 (round to nearest even).  A row
 * whose V(b,i) is empty gets O = 0 exactly and LSE = -inf (TileOPs
 * MHADecodePagedWithKVCacheFwdOp / GQAPagedFwdOp: "outputs zeros"; MATE "QSA",
 * Core Attention: empty rows give -inf LSE).  LSE is the natural-log
 * log-sum-exp of the scaled logits of the row, FP32 (MATE "QSA", Core
 * Attention: natural-log LSE shaped like the query without its last axis).
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers of the current CUDA device,
 *     row-major, contiguous, in BSHD order (batch, sequence, head, head_dim),
 *     head_dim contiguous (TileOPs GQADenseFwdOp, forward).  bfloat16 data is
 *     passed as raw 16-bit storage (void*).
 *   - q, k, v, o must be 16-byte aligned; paged caches too.
 *   - The caller owns every buffer (inputs, outputs, workspace).  The library
 *     allocates no device memory on these paths and never reads device data
 *     back to the host; work is enqueued on `stream` and returns immediately.
 *   - Inputs are read only (RL-Kernel: "no in-place mutation").
 *   - Argument checks run on the host before any launch; a failed check
 *     launches nothing and returns the status.  A launch failure returns
 *     GQA_ERR_CUDA.
 *   - D (head_dim) must be 64, 128 or 256; Hq must be a multiple of Hkv
 *     (RL-Kernel, Known Limitations: ValueError otherwise).
 */
#ifndef GQA_ATTN_H
#define GQA_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the runtime and driver stream handle types are the same). */
typedef struct CUstream_st* gqa_stream_t;

typedef enum {
    GQA_OK = 0,
    GQA_ERR_INVALID_ARG = 1,  /* a size or pointer argument is out of range */
    GQA_ERR_UNSUPPORTED = 2,  /* a valid combination the library has no kernel for */
    GQA_ERR_MISALIGNED = 3,   /* a pointer is not 16-byte aligned */
    GQA_ERR_WORKSPACE = 4,    /* workspace missing or smaller than required */
    GQA_ERR_CUDA = 5,         /* a CUDA call or kernel launch failed */
    GQA_ERR_TIMEOUT = 6       /* a kernel gave up waiting (see gqa_device_error) */
} gqa_status;

/*
 * Optional terms of a call (TileOPs "Attention Operators", GQADenseFwdOp stages
 * 5-6, and GQAPagedFwdOp's sinks).  Pass NULL for none; a zeroed struct with
 * both windows at -1 is the same.
 *   window_left   keys admitted left of the query's key position p_i (key j is
 *                 visible only if j >= p_i - window_left); -1 = unlimited
 *   window_right  keys admitted right of p_i (j <= p_i + window_right); -1 =
 *                 unlimited; with the causal mask (j <= p_i already) a
 *                 window_right >= 0 changes nothing
 *   softcap       c > 0 replaces each visible scaled score z with c*tanh(z/c);
 *                 0 disables capping; negative or non-finite is refused
 *   sinks         NULL, or a DEVICE array of Hq float32 logits, one per query
 *                 head, that join the softmax denominator only (not scaled,
 *                 not capped): weight_j = exp(z_j) / (sum_j exp(z_j) +
 *                 exp(sink_h)); the LSE includes exp(sink_h).  -inf disables a
 *                 sink; +inf makes that head's output zero (LSE +inf).  A row
 *                 with no visible key outputs zeros with LSE -inf either way.
 *                 4-byte aligned; read on the device, never copied.
 *   dtype         GQA_BF16 (default) or GQA_FP16 (TileOPs GQAPagedFwdOp serves
 *                 "a float16 or bfloat16 dtype" shared by Q and the cache):
 *                 q, k, v / the caches and o all have this type; products and
 *                 sums stay FP32, P is rounded to the same type before P V.
 * Window values below -1, a bad softcap or another dtype return
 * GQA_ERR_INVALID_ARG.
 */
/* Element type of q, k, v (or the caches) and o. */
typedef enum { GQA_BF16 = 0, GQA_FP16 = 1 } gqa_dtype;

typedef struct {
    int window_left;
    int window_right;
    float softcap;
    const float* sinks;
    int dtype;            /* gqa_dtype: every 16-bit tensor of the call; 0 = bfloat16 */
} gqa_options;

/*
 * Dense prefill / chunked prefill (TileOPs GQADenseFwdOp; RL-Kernel
 * "Prefill / Decode / KV-cache Shared Contract": one expression covers
 * Sq == Skv, chunked prefill and Sq < Skv).
 *
 *   q    [B, Sq,  Hq,  D] bf16        k, v [B, Skv, Hkv, D] bf16
 *   key_padding_mask  [B, Skv] bytes, nonzero = keep, or NULL for none
 *                     (RL-Kernel Tensor Contract: False columns become -inf)
 *   o    [B, Sq, Hq, D] bf16 (written)
 *   lse  [B, Sq, Hq] float (written), or NULL to skip it
 *   causal  nonzero applies the end-aligned causal mask
 *   scale   the score multiplier; the library takes it as given (0.0 included);
 *           callers wanting the default pass 1/sqrt(D)
 *
 * B, Hq, Hkv, D > 0; Sq >= 0, Skv >= 0.  Sq > Skv with causal is accepted:
 * rows i < Sq - Skv see no key and get zeros.  Skv == 0 gives all-zero O.
 * D = 64 and 128 run two 128-row query tiles per CTA; D = 256 (the 24/2/D256
 * geometry of MATE "QSA") one tile per CTA with double-buffered scores.
 */
gqa_status attn_fwd_dense(const void* q, const void* k, const void* v,
                          const uint8_t* key_padding_mask, void* o, float* lse,
                          int B, int Hq, int Hkv, int Sq, int Skv, int D,
                          int causal, float scale, gqa_stream_t stream);

/* attn_fwd_dense with optional terms (opts may be NULL). */
gqa_status attn_fwd_dense_ex(const void* q, const void* k, const void* v,
                             const uint8_t* key_padding_mask, void* o, float* lse,
                             int B, int Hq, int Hkv, int Sq, int Skv, int D,
                             int causal, float scale, const gqa_options* opts,
                             gqa_stream_t stream);

/*
 * Paged decode (TileOPs MHADecodePagedWithKVCacheFwdOp and GQAPagedFwdOp;
 * split-KV with an LSE merge as in MATE "QSA", Core Attention).
 *
 *   q        [B, Sq, Hq, D] bf16  (Sq new query tokens per request)
 *   k_cache, v_cache  [num_pages, page_size, Hkv, D] bf16
 *   real_seqlen_kv    [B] int32: request b's cache length L_b, its Sq query
 *                     tokens included; 0 <= L_b <= max_pages * page_size
 *   block_table       [B, max_pages] int32: logical page p of request b lives
 *                     in physical page block_table[b, p]; token t is slot
 *                     t % page_size of page block_table[b, t / page_size]
 *   o        [B, Sq, Hq, D] bf16 (written); lse [B, Sq, Hq] float or NULL
 *   causal   nonzero: query i sees keys t <= i + L_b - Sq
 *   workspace / workspace_bytes: device scratch of at least
 *            attn_decode_paged_workspace_size(...) bytes, 256-byte aligned;
 *            its contents on entry do not matter; calls that share one
 *            workspace must not overlap on the GPU.
 *
 * Caller obligations (attn_validate_paged checks them on the host): the
 * entries block_table[b, 0 .. ceil(L_b / page_size) - 1] lie in
 * [0, num_pages); later entries are never read (-1 is fine there).  The
 * device does not report violations, but it never dereferences a page id
 * outside [0, num_pages) (such rows read as zeros) and clamps lengths to
 * [0, max_pages * page_size], so no memory outside the pool is touched; the
 * results of such requests are unspecified.  num_pages * page_size must stay
 * below 2^31 (GQA_ERR_UNSUPPORTED otherwise).
 */
gqa_status attn_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* real_seqlen_kv, const int32_t* block_table,
                             int page_size, void* o, float* lse,
                             int B, int Sq, int Hq, int Hkv, int D,
                             int num_pages, int max_pages, int causal, float scale,
                             void* workspace, size_t workspace_bytes,
                             gqa_stream_t stream);

/*
 * attn_decode_paged with optional terms (opts may be NULL).  A left window
 * also bounds what is read: keys left of every query's window are not loaded.
 * Same workspace size.
 */
gqa_status attn_decode_paged_ex(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* real_seqlen_kv, const int32_t* block_table,
                                int page_size, void* o, float* lse,
                                int B, int Sq, int Hq, int Hkv, int D,
                                int num_pages, int max_pages, int causal, float scale,
                                const gqa_options* opts, void* workspace, size_t workspace_bytes,
                                gqa_stream_t stream);

/*
 * Paged decode over float8_e4m3fn key and value caches (TileOPs "Attention
 * Operators", GQADenseFwdOp stage 2, FP8 dequantization, and GQAVarlenFwdOp's
 * one scale per request and KV head): key t of KV head r in request b is
 * K * k_scale[b * Hkv + r], its value V * v_scale[b * Hkv + r]; Q is 16-bit.
 * The result is the attn_decode_paged_ex definition on those keys and values.
 *
 *   k_cache, v_cache  [num_pages, page_size, Hkv, D] e4m3fn bytes (sign, 4
 *                     exponent bits with bias 7, 3 mantissa bits; 0x7F and 0xFF
 *                     are NaN and must not occur), 16-byte aligned
 *   k_scale, v_scale  [B, Hkv] float device arrays, or NULL for all ones;
 *                     every scale finite and positive, a caller obligation as
 *                     in TileOPs "Attention Operators",
 *                     GQAPrefillPagedWithKVCacheFwdOp (validate_inputs): the
 *                     library reads them on the GPU only and does not check
 *                     them; another value corrupts the rows of that request
 *                     and KV head
 *   q, o              16-bit: bfloat16, or float16 with opts->dtype = GQA_FP16
 *   other arguments   as attn_decode_paged_ex; the same workspace size
 *                     (attn_decode_paged_workspace_size) is enough.
 *
 * The keys and values are widened exactly to float16 on the GPU and the
 * products run in float16 with FP32 accumulation, so Q is rounded to float16
 * once: a bfloat16 Q keeps every bit for magnitudes in [2^-14, 65504] and must
 * stay below 65504.  Supported: D = 128 or 256 (GQA_ERR_UNSUPPORTED
 * otherwise) and any page size: pages that are a multiple of 8 and divide,
 * or are divided by, the key tile (64 tokens at D = 128, 32 at D = 256) move
 * by TMA, other sizes are gathered row by row (slower loads, the same
 * results; KV groups of 32 or more rows then take the split kernel).  Caller
 * obligations and the handling of bad page ids and lengths are those of
 * attn_decode_paged.
 */
gqa_status attn_decode_paged_fp8kv(const void* q, const void* k_cache, const void* v_cache,
                                   const float* k_scale, const float* v_scale,
                                   const int32_t* real_seqlen_kv, const int32_t* block_table,
                                   int page_size, void* o, float* lse,
                                   int B, int Sq, int Hq, int Hkv, int D,
                                   int num_pages, int max_pages, int causal, float scale,
                                   const gqa_options* opts, void* workspace, size_t workspace_bytes,
                                   gqa_stream_t stream);

/*
 * Bytes of workspace attn_decode_paged needs for these sizes on the current
 * device (0 for invalid sizes).  A pure function of its arguments and the
 * device's SM count.
 */
size_t attn_decode_paged_workspace_size(int B, int Sq, int Hq, int Hkv, int D,
                                        int page_size, int max_pages);

/*
 * Paged decode that allocates nothing and takes no workspace.  The pages this
 * library follows have no counterpart of it; it exists for callers that
 * cannot allocate device memory or hand over a workspace (a serving engine
 * whose memory is all pre-reserved by its own pool, a plugin inside a host
 * framework that forbids allocation while it runs, a latency-critical loop
 * that cannot pay for cudaMalloc's implicit synchronisation).
 *
 * Same arguments, semantics and checks as attn_decode_paged, without
 * `workspace` / `workspace_bytes`: the split-KV partials live in a fixed
 * device array inside the library of attn_decode_paged_noalloc_max_workspace()
 * bytes (32 MiB), which every GPU that loads the library holds until the
 * process exits.  Sizes needing more than that (see
 * attn_decode_paged_workspace_size) return GQA_ERR_WORKSPACE and launch
 * nothing.  The first call on a device looks up the array's device address
 * with that device current; make that first call before any stream capture.
 * All calls share the array: calls whose kernels overlap on the GPU (for
 * example on two streams) race; nothing in it needs clearing between calls.
 * No cudaMalloc, cudaFree or allocating library routine is called.
 */
gqa_status attn_decode_paged_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* real_seqlen_kv, const int32_t* block_table,
                                     int page_size, void* o, float* lse,
                                     int B, int Sq, int Hq, int Hkv, int D,
                                     int num_pages, int max_pages, int causal, float scale,
                                     gqa_stream_t stream);

/* Bytes of the fixed device array attn_decode_paged_noalloc uses. */
size_t attn_decode_paged_noalloc_max_workspace(void);

/*
 * Packed variable-length attention (TileOPs "Attention Operators",
 * GQAVarlenFwdOp), one launch for any mix of request lengths.
 *
 *   q    [total_q, Hq, D]    k, v  [total_kv, Hkv, D]     (THD, 16-bit)
 *   cu_seqlens_q, cu_seqlens_kv  [B + 1] int32 device offsets: request b
 *        owns query rows [cu_seqlens_q[b], cu_seqlens_q[b + 1]) and key /
 *        value rows [cu_seqlens_kv[b], cu_seqlens_kv[b + 1]); a request may
 *        have no query row or no key
 *   o    [total_q, Hq, D] (written); lse [total_q, Hq] float or NULL
 *   causal  nonzero: query i of request b sees its keys j <= i + Skv_b - Sq_b
 *   opts    window, softcap, sinks and dtype as for attn_fwd_dense_ex
 *   workspace / workspace_bytes: device scratch of at least
 *        attn_varlen_workspace_size(B, total_q, Hq, Hkv) bytes, 16-byte
 *        aligned; calls that share one must not overlap on the GPU.
 *
 * The offsets stay on the device (no host read-back; the call can be
 * captured in a CUDA graph with the offsets as live inputs).  The caller
 * guarantees cu[0] = 0, non-decreasing offsets and cu[B] = total; the device
 * clamps every offset into [0, total], so malformed offsets give wrong
 * results but no access outside q, k, v, o and lse; query rows outside every
 * request are not written.  The g = Hq / Hkv query heads of a KV group share
 * one tile (g <= 128, GQA_ERR_UNSUPPORTED otherwise).
 */
gqa_status attn_fwd_varlen(const void* q, const void* k, const void* v,
                           const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                           void* o, float* lse, int B, int total_q, int total_kv,
                           int Hq, int Hkv, int D, int causal, float scale,
                           const gqa_options* opts, void* workspace, size_t workspace_bytes,
                           gqa_stream_t stream);

/*
 * Packed queries over a paged cache (TileOPs "Attention Operators",
 * GQAPagedFwdOp): prefill chunks and decode steps of many requests in one
 * launch.
 *
 *   q    [total_q, Hq, D]; request b owns rows [cu_seqlens_q[b], cu_seqlens_q[b + 1])
 *   k_cache, v_cache  [num_pages, page_size, Hkv, D]
 *   cache_seqlens     [B] int32: request b's cache length L_b, its query
 *                     tokens included; query i of request b sits at key
 *                     position i + L_b - Sq_b
 *   block_table       [B, max_pages] int32, as for attn_decode_paged
 *   o    [total_q, Hq, D] (written); lse [total_q, Hq] float or NULL
 *   workspace         at least attn_varlen_workspace_size(B, total_q, Hq, Hkv)
 *                     bytes, 16-byte aligned.  With
 *                     attn_paged_workspace_size(B, total_q, Hq, Hkv, D,
 *                     page_size, max_pages) bytes, 256-byte aligned, the
 *                     requests with exactly one query (decode steps) run on
 *                     the split-KV decode kernel of attn_decode_paged (where
 *                     Hq / Hkv < 32) and the rest on the packed kernel; with
 *                     less, every request runs on the packed kernel.  Results
 *                     agree within the usual tolerance either way.  Calls
 *                     sharing a workspace must not overlap on the GPU.
 *
 * Streams: with the decode steps on the split kernel, the packed kernel runs
 * beside them on a second stream of the highest priority that the library
 * keeps per device and host thread (created on the first such call that is
 * not inside a stream capture), forked from `stream` after the plan kernel
 * and joined back into `stream` with events before the call returns: work
 * queued on `stream` afterwards sees both parts complete, and a captured call
 * records the fork and join in the graph.  The packed kernel then keeps the
 * share of the SMs that the plan kernel estimates, on the device, from the
 * requests' lengths; the decode CTAs take the rest.  If the second stream
 * cannot be had, both parts run one after the other on `stream`.
 *
 * Any page_size >= 1 and num_pages >= 1: pages whose size is a multiple of 8
 * move as 8-row TMA blocks, other page sizes are gathered row by row (slower
 * loads, the same results).  Caller obligations on the
 * table as for attn_decode_paged; lengths are clamped to
 * [0, max_pages * page_size] and a page id outside [0, num_pages) reads as
 * zeros.  Cache slots past L_b and pages past a request's end never reach
 * the result.
 */
gqa_status attn_fwd_paged(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* cu_seqlens_q, const int32_t* cache_seqlens,
                          const int32_t* block_table, int page_size, void* o, float* lse,
                          int B, int total_q, int Hq, int Hkv, int D, int num_pages,
                          int max_pages, int causal, float scale, const gqa_options* opts,
                          void* workspace, size_t workspace_bytes, gqa_stream_t stream);

/* Workspace bytes of attn_fwd_varlen / attn_fwd_paged (0 for invalid sizes). */
size_t attn_varlen_workspace_size(int B, int total_q, int Hq, int Hkv);

/*
 * Workspace bytes of attn_fwd_paged with its single-query requests on the
 * split-KV decode kernel: the packed plan's bytes, then, from a 256-byte
 * boundary, the split partials of B one-query requests (attn_decode_paged's
 * workspace for Sq = 1).  Equals attn_varlen_workspace_size when the sizes
 * keep every request on the packed kernel; 0 for invalid sizes.
 */
size_t attn_paged_workspace_size(int B, int total_q, int Hq, int Hkv, int D, int page_size, int max_pages);

/*
 * Optional host-side check of the paged metadata (the TileOPs
 * validate_inputs=True analogue).  Copies real_seqlen_kv and block_table to
 * the host (synchronising `stream`) and checks every length and every needed
 * table entry.  Returns GQA_OK or GQA_ERR_INVALID_ARG.  Not for the hot path.
 */
gqa_status attn_validate_paged(const int32_t* real_seqlen_kv, const int32_t* block_table,
                               int B, int Sq, int page_size, int num_pages, int max_pages,
                               int causal, gqa_stream_t stream);

/* Static description of a status code. */
const char* gqa_status_string(gqa_status status);

/*
 * Every wait inside the kernels is bounded; a wait that runs out records a
 * code in a device-side word and the kernel returns early.  This call
 * synchronises the device, returns GQA_ERR_TIMEOUT if the word is set
 * (clearing it) and GQA_OK otherwise.  Diagnostic, not for the hot path.
 */
gqa_status gqa_device_error(void);

/* Library version string. */
const char* gqa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_H */
