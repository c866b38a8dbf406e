/*
 * paged_attn.h - C ABI of the GB300 (sm_103a) paged-KV decode attention library.
 *
 * The operation (ATOM model-operations guide, "Multi-head attention": forward
 * flow step 3 and the "Attention dispatch" table, decode rows; configuration
 * guide, "Quick reference": kv_cache_block_size = 16, kv_cache_dtype bf16|fp8;
 * high-interactivity blog, "Attention Decode: Split Memory Work to Fill the
 * Device"): every query token of every sequence, for every query head hq,
 * attends over the sequence's cached keys and values,
 *
 *     out[t, hq, :] = sum_j softmax_j(scale * <q[t, hq, :], K_j>) * V_j
 *     lse[t, hq]    = ln sum_j exp(scale * <q[t, hq, :], K_j>)
 *
 * where K_j, V_j are the rows of KV head hk = hq / (Hq / Hkv) for logical
 * token j, found at physical page block_tables[i][j / 16], slot j % 16.
 * Sequence i has L_i = seq_lens[i] cached tokens, which include its own q_i
 * query tokens; query token r (0 <= r < q_i) sees keys j <= L_i - q_i + r
 * (causal inside a multi-token verification run, as in MTP speculative
 * decoding; a single-token decode sees all L_i keys).  fp8 caches hold OCP
 * e4m3fn codes; the value of a cached K element is code * k_scale and of a V
 * element code * v_scale (one fp32 scale per tensor).  bf16 caches ignore
 * k_scale and v_scale.
 *
 * Conventions for every entry point:
 *   - All tensor data pointers are DEVICE pointers on the current CUDA device.
 *   - Strides are in elements.  Shapes and strides are read on the host only;
 *     the library never reads device memory on the host and never
 *     synchronises the stream.  Work is enqueued asynchronously on `stream`.
 *   - The caller owns every tensor and must keep it alive until the stream
 *     work completes.  The library owns only a per-device split workspace
 *     (grown on demand outside stream capture, see paged_attn_reserve) unless
 *     the caller passes its own through pa_options_t.
 *   - Functions return a pa_status (PA_OK = 0); nothing throws across the
 *     ABI.  paged_attn_last_error_message() gives a human-readable detail of
 *     the last failure on the calling thread.
 *   - The first call of any entry point on a device sets that device up once
 *     (attributes, kernel limits, the device addresses of the status word and
 *     of the no-allocation scratch array).  The library keeps that state for
 *     the life of the process and does not survive cudaDeviceReset: after a
 *     reset, every later call on that device is undefined.
 */
#ifndef PAGED_ATTN_H
#define PAGED_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same underlying type as cudaStream_t / CUstream; NULL = legacy default stream. */
typedef struct CUstream_st* pa_stream_t;

/* Element types of pa_tensor_t. */
enum pa_dtype {
  PA_BF16 = 1,      /* bfloat16                                  */
  PA_FP8_E4M3 = 2,  /* OCP fp8 e4m3fn codes (1 byte per element) */
  PA_F32 = 3,       /* float32                                   */
  PA_I32 = 4        /* int32                                     */
};

/* Status codes. */
enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,  /* shape, dtype, stride or alignment mismatch; NULL required pointer */
  PA_ERR_UNSUPPORTED = 2,  /* valid but outside the kernel's envelope (head_dim, group size, ...) */
  PA_ERR_WORKSPACE = 3,    /* workspace too small while the stream is being captured, or caller
                              workspace too small */
  PA_ERR_CUDA = 4          /* a CUDA runtime/driver call or a kernel launch failed */
};

/* A strided view of device memory (DLPack-like, without the dependency).
 * Dimensions beyond ndim are ignored. */
typedef struct pa_tensor_t {
  void* data;
  int32_t dtype;      /* enum pa_dtype */
  int32_t ndim;
  int64_t shape[4];
  int64_t stride[4];  /* elements */
} pa_tensor_t;

/* Optional controls for paged_attn_decode_ex.  Zero-initialise for defaults. */
typedef struct pa_options_t {
  int32_t num_ctas;            /* >0: launch this many split CTAs instead of one per SM */
  int32_t min_pages_per_cta;   /* >0: override the minimum pages of work per CTA (default 4) */
  int32_t heads_per_cta;       /* >0: KV heads per CTA (must divide Hkv); 0 = planner's choice */
  int32_t disable_pdl;         /* !=0: launch both kernels without programmatic dependent launch */
  int32_t page_pairing;        /* 0: planner's choice; 1: never; 2: always process two pages at once */
  int32_t sliding_window;      /* W > 0: query at position p sees only keys p-W < j <= p (the pages'
                                  sliding_window; <= 0 = off); pages wholly before the window are
                                  never read */
  const void* sinks;           /* optional device pointer to float[Hq]: per-query-head attention sink
                                  logits (GPT-OSS style): each joins its row's softmax normaliser with
                                  a zero value row and is included in lse; NULL = none */
  void* workspace;             /* optional caller-owned device workspace ...                   */
  size_t workspace_bytes;      /* ... of this size (see paged_attn_workspace_size)            */
  void* split_start_event;     /* optional cudaEvent_t recorded just before the split kernel  */
  void* split_stop_event;      /* optional cudaEvent_t recorded just after the split kernel   */
  int32_t use_tcgen05;         /* split kernel: 0 = planner's choice (the tensor-memory kernel when
                                  G * max_query_len > 64, else the mma.sync kernel); 1 = never
                                  (PA_ERR_UNSUPPORTED above 64 rows); 2 = always (bf16 caches only) */
  const struct pa_tensor_t* k_token_scales;  /* optional per-token scales of an fp8 cache (the pages'
                                  reshape_and_cache_with_pertoken_quant layout: one fp32 scale per
                                  cached row): f32 [NB, Hkv, 16], entry [page][head][slot];
                                  stride[2] == 1, stride[1] == 16, stride[0] % 4 == 0, data 16-byte
                                  aligned.  A cached K element's value is then
                                  code * k_scale * k_token_scales[page][head][slot] (pass k_scale =
                                  1 for a purely per-token cache).  NULL (or data NULL) = none.
                                  Requires v_token_scales too and an fp8 cache; entries of slots
                                  past a sequence's end may hold anything, even non-finite values */
  const struct pa_tensor_t* v_token_scales;  /* the same for V (value = code * v_scale * scale) */
  int32_t wait_limit_us;       /* >0: every pipeline wait inside the decode kernels gives up after this
                                  many microseconds (status bit 3, the kernel returns); 0 = 2 seconds */
  int32_t test_starve_cta;     /* testing aid for the give-up path, 0 = off.  k > 0: the producer warp
                                  of split CTA k-1 issues no copies, so that CTA's consumer warps wait
                                  out wait_limit_us, set status bit 3 and return; the call's results
                                  are then undefined (the affected rows keep stale partials).  The
                                  mma.sync split kernel only (PA_ERR_UNSUPPORTED for the tcgen05 and
                                  MLA kernels) */
  int32_t segment_cost_pages;  /* tensor-memory MLA kernel: the work split charges
                                  every unit (sequence, head chunk) a CTA starts this many pages on
                                  top of its pages, so CTAs that open more units get fewer pages
                                  (a unit costs a Q staging and an epilogue).  0 = the planner's
                                  value for the shape; < 0 = an equal page split.  Ignored by the
                                  other kernels */
} pa_options_t;

/* Launch plan the library picks for a problem shape (for tests, tuning and
 * roofline accounting). */
typedef struct pa_plan_t {
  int32_t num_ctas;          /* split-kernel grid size                                  */
  int32_t heads_per_cta;     /* KV heads a CTA processes per page (HC)                  */
  int32_t row_tiles;         /* 16-row tiles per KV head (ceil(G*max_query_len/16); 8 for tcgen05) */
  int32_t num_stages;        /* depth of the shared-memory page ring                    */
  int32_t threads_per_cta;   /* 32 * (1 producer + heads_per_cta * row_tiles); tcgen05: 384 */
  int32_t smem_bytes;        /* dynamic shared memory per CTA                           */
  int32_t min_pages_per_cta; /* work below which fewer CTAs are used                    */
  int32_t merge_rows;        /* rows per merge unit (heads_per_cta * G * max_query_len) */
  int32_t page_pairing;      /* 1 if consumer warps take two pages of a sequence at once */
  int64_t workspace_bytes;   /* split workspace the call needs                          */
  int32_t variant;           /* 0: mma.sync warps; 1: tcgen05 / tensor-memory kernel; 2: MLA on
                                mma.sync warps; 3: MLA on tcgen05 / tensor memory           */
  int32_t block_pages;       /* pages a consumer step takes (1, 2 paired, 4 tcgen05)    */
} pa_plan_t;

/*
 * paged_attn_decode - decode attention over a paged KV cache (definition above).
 *
 *   q               bf16 [T, Hq, D]; stride[2] == 1, stride[1] == D, stride[0]*2 % 16 == 0,
 *                   data 16-byte aligned.  T = total query tokens.
 *   k_cache         bf16 or fp8e4m3 [NB, 16, Hkv, D]; stride[3] == 1; every other stride
 *                   times the element size a multiple of 16 bytes; data 16-byte aligned.
 *   v_cache         same dtype and shape as k_cache (strides may differ, same rules).
 *   block_tables    int32 [B, max_blocks]; stride[1] == 1.  Entry [i][j] is the physical
 *                   page of logical page j of sequence i; only j < ceil(L_i / 16) is read.
 *   seq_lens        int32 [B], contiguous.  L_i >= q_i >= 1.
 *   query_start_loc int32 [B+1] contiguous cumulative query-token offsets (ragged MTP
 *                   runs), or data == NULL: one query token per sequence (T == B).
 *   max_query_len   host-known upper bound of q_i (1 when query_start_loc is NULL);
 *                   chooses the tile without a device read.  G * max_query_len <= 128
 *                   for bf16 caches (above 64 rows the tcgen05 / tensor-memory kernel
 *                   runs), <= 64 for fp8 caches.
 *   scale           softmax scale applied to <q, k> (e.g. 1/sqrt(D)).
 *   k_scale, v_scale per-tensor dequantisation scales of fp8 caches (ignored for bf16).
 *   out             bf16 [T, Hq, D], stride[2] == 1; written.
 *   lse             f32 [T, Hq] natural-log log-sum-exp of the scaled logits, or
 *                   data == NULL (not written).
 *   stream          stream the work is enqueued on.
 *
 * Supported: D in {64, 128}; page size 16; Hq % Hkv == 0; 1 <= B <= 8192.
 * Errors: PA_ERR_INVALID_ARG / PA_ERR_UNSUPPORTED are detected on the host before
 * anything is enqueued.  Data errors that only the device can see (a page id
 * outside [0, NB), L_i < q_i, q_i > max_query_len) set bits of the device status
 * word (paged_attn_device_status); the affected rows are undefined.
 */
int paged_attn_decode(const pa_tensor_t* q, const pa_tensor_t* k_cache, const pa_tensor_t* v_cache,
                      const pa_tensor_t* block_tables, const pa_tensor_t* seq_lens,
                      const pa_tensor_t* query_start_loc, int32_t max_query_len, float scale,
                      float k_scale, float v_scale, const pa_tensor_t* out, const pa_tensor_t* lse,
                      pa_stream_t stream);

/* paged_attn_decode with options (opts may be NULL = defaults).  Same operation,
 * arguments and errors as paged_attn_decode. */
int paged_attn_decode_ex(const pa_tensor_t* q, const pa_tensor_t* k_cache, const pa_tensor_t* v_cache,
                         const pa_tensor_t* block_tables, const pa_tensor_t* seq_lens,
                         const pa_tensor_t* query_start_loc, int32_t max_query_len, float scale,
                         float k_scale, float v_scale, const pa_tensor_t* out, const pa_tensor_t* lse,
                         const pa_options_t* opts, pa_stream_t stream);

/*
 * paged_attn_decode_static_scratch - paged_attn_decode for callers that cannot
 * allocate device memory.  The pages have no counterpart to this entry point.
 *
 * Same operation, arguments, layouts and errors as paged_attn_decode, but the
 * split scratch comes from a fixed 16 MiB (16777216-byte) array compiled into
 * the library's device code, so the call never calls cudaMalloc/cudaFree or any
 * other allocating routine.  It serves callers whose memory is owned by a pool
 * or allocator they must not bypass, or that run where allocation is not
 * allowed.
 *   - The library's per-device set-up (the first call of ANY entry point on a
 *     device, with that device current) looks up the array's device address,
 *     which also loads it under CUDA's lazy module loading; from then on that
 *     GPU holds the 16 MiB until the process exits.  Make one call on each
 *     device before a memory pool takes the device's free memory, and before
 *     any stream capture.
 *   - A shape needing more scratch than 16 MiB (see paged_attn_workspace_size)
 *     is rejected with PA_ERR_WORKSPACE before anything is enqueued.
 *   - All calls share the one array and it keeps the last call's contents (no
 *     part of it needs to start at zero); calls whose GPU work overlaps, e.g. on
 *     two streams at once, race on it and must be serialised by the caller.
 */
int paged_attn_decode_static_scratch(const pa_tensor_t* q, const pa_tensor_t* k_cache,
                                     const pa_tensor_t* v_cache, const pa_tensor_t* block_tables,
                                     const pa_tensor_t* seq_lens, const pa_tensor_t* query_start_loc,
                                     int32_t max_query_len, float scale, float k_scale, float v_scale,
                                     const pa_tensor_t* out, const pa_tensor_t* lse, pa_stream_t stream);

/*
 * paged_attn_cache_write - write new tokens' K and V rows into the paged caches
 * (ATOM model-operations guide, "KV cache operations": standard (bf16) and FP8
 * KV cache write; token_layout/slots.py: slot_mapping, "which KV slot a token is
 * written to").
 *
 *   key, value      bf16 [T, Hkv, D]; stride[2] == 1, other strides multiples of 8
 *                   elements, data 16-byte aligned.
 *   slot_mapping    int32 [T] contiguous.  Token t goes to page slot_mapping[t] / 16,
 *                   slot slot_mapping[t] % 16; a negative entry (padding) writes
 *                   nothing; an entry >= 16 * NB writes nothing and sets bit 0 of the
 *                   device status word.  Two tokens with the same slot: which one
 *                   lands is unspecified.
 *   k_cache, v_cache bf16 or fp8e4m3 [NB, 16, Hkv, D]: stride[3] == 1, other
 *                   strides multiples of 16 bytes, data 16-byte aligned.  D is any
 *                   multiple of 8 up to 512 (of 16 for fp8 caches, by the stride
 *                   rule), Hkv at most 4096, T at most 2^30, NB below 2^31
 *                   (else PA_ERR_UNSUPPORTED).  The decode entry points read
 *                   D = 64 and 128.
 *   k_scale, v_scale fp8 caches only: the stored code is e4m3fn(x / scale), one
 *                   IEEE fp32 division (a cached value reads back as code * scale);
 *                   round to nearest even, finite magnitudes above 448 and
 *                   infinities saturate to +-448.  bf16 caches store x unchanged.
 *   stream          stream the work is enqueued on.
 *
 * Errors as for paged_attn_decode.  Asynchronous; allocates nothing.
 */
int paged_attn_cache_write(const pa_tensor_t* key, const pa_tensor_t* value, const pa_tensor_t* slot_mapping,
                           const pa_tensor_t* k_cache, const pa_tensor_t* v_cache, float k_scale, float v_scale,
                           pa_stream_t stream);

/*
 * paged_attn_cache_write_per_token - the fp8 KV-cache write with one scale per
 * written row (ATOM model-operations guide, "KV cache operations": FP8 KV cache
 * write, aiter.reshape_and_cache_with_pertoken_quant; the attention-dispatch
 * note that per-token quantised layers carry more than one descale per tensor).
 *
 *   key, value, slot_mapping  as for paged_attn_cache_write.
 *   k_cache, v_cache          fp8e4m3 [NB, 16, Hkv, D] (bf16 caches are rejected).
 *   k_token_scales, v_token_scales  f32 [NB, Hkv, 16], any non-negative strides,
 *                   4-byte aligned: entry [page][head][slot] receives the row's scale.
 *   For every written (token, head) row x (bf16, D values): amax = max_d |x_d|;
 *   scale = amax / 448 and code_d = e4m3fn(x_d / scale), both IEEE fp32
 *   divisions (the row reads back as code * scale), round to nearest even,
 *   saturating to +-448; an all-zero row (+0 or -0 elements) stores scale 0 and
 *   the code 0x00 throughout.  Rows must be finite.
 *   paged_attn_decode_ex reads such a cache with pa_options_t.k_token_scales /
 *   v_token_scales and k_scale = v_scale = 1.
 *
 * Errors, padding slots and out-of-range slots as for paged_attn_cache_write.
 * Asynchronous; allocates nothing.
 */
int paged_attn_cache_write_per_token(const pa_tensor_t* key, const pa_tensor_t* value,
                                     const pa_tensor_t* slot_mapping, const pa_tensor_t* k_cache,
                                     const pa_tensor_t* v_cache, const pa_tensor_t* k_token_scales,
                                     const pa_tensor_t* v_token_scales, pa_stream_t stream);

/*
 * paged_attn_mla_decode - multi-head latent attention (MLA) decode over a paged
 * latent cache (ATOM model-operations guide, "Multi-head latent attention
 * (attention_mla.py)": MLAModules kv_lora_rank / qk_rope_head_dim, decode flow
 * step 2, mla_decode_fwd after fused_qk_rope_concat_and_cache_mla; high-
 * interactivity blog, "Attention Decode" (MLA split count, fp32 per-split
 * log-sum-exp) and "Multi-Token Prediction" (query length four)).
 *
 * Each cached token is one row C_j = [c_kv (kv_lora_rank) | k_pe (rope)] shared by
 * every query head; the query arrives absorbed (q_nope times the K up-projection,
 * then q_pe), as wide as a cached row.  For query token t of sequence i (query row r
 * of its run, position p = L_i - q_i + r) and head h:
 *
 *     s_j          = scale * <q[t, h, :], C_j>                     j = 0 .. p
 *     out[t, h, :] = sum_j softmax_j(s) * C_j[0 : kv_lora_rank]    (latent space)
 *     lse[t, h]    = ln sum_j exp(s_j)
 *
 * with C_j found at page block_tables[i][j / 16], slot j % 16.  An fp8 cache holds
 * e4m3fn codes; an element's value is code * kv_scale in the logit and in the output.
 *
 *   q               bf16 [T, Hq, 576] (kv_lora_rank 512 + rope 64); stride[2] == 1,
 *                   stride[1] == 576, stride[0] * 2 % 16 == 0, data 16-byte aligned.
 *   kv_cache        bf16 or fp8e4m3 [NB, 16, 576]; stride[2] == 1, other strides times
 *                   the element size multiples of 16 bytes, data 16-byte aligned.
 *   block_tables, seq_lens, query_start_loc, max_query_len   as for paged_attn_decode;
 *                   the query heads of one sequence form Hq * max_query_len rows per
 *                   latent row, processed in chunks of at most 32 rows (max_query_len
 *                   <= 32).
 *   scale           softmax scale (e.g. 1/sqrt(qk_nope_head_dim + qk_rope_head_dim)).
 *   kv_scale        fp8 caches: dequantisation scale (ignored for bf16).
 *   out             bf16 [T, Hq, 512]; stride[2] == 1, other strides multiples of 4.
 *   lse             f32 [T, Hq] or data == NULL.
 *   opts            (the _ex form) num_ctas, min_pages_per_cta, disable_pdl,
 *                   workspace / workspace_bytes, wait_limit_us and the split events
 *                   apply; use_tcgen05 picks the split kernel (0: the planner's
 *                   choice, the tensor-memory kernel for fp8 caches or units of
 *                   more than 16 rows, else the mma.sync kernel; 1: always the
 *                   mma.sync kernel; 2: always the tensor-memory kernel);
 *                   segment_cost_pages tunes the tensor-memory kernel's work
 *                   split; the grouped-query
 *                   options (heads_per_cta, sliding_window, sinks, token scales,
 *                   test_starve_cta) are rejected with PA_ERR_UNSUPPORTED.
 *
 * Errors, device status bits, workspace and graph-capture rules as for
 * paged_attn_decode (paged_attn_mla_workspace_size gives the workspace a shape needs).
 * The pieces of a sequence cut across CTAs meet in f16 (their normalised outputs):
 * cached values must lie within the f16 range (|v| <= 65504; any fp8 cache does);
 * an overflow sets status bit 4 and the affected rows are undefined.
 */
int paged_attn_mla_decode(const pa_tensor_t* q, const pa_tensor_t* kv_cache, const pa_tensor_t* block_tables,
                          const pa_tensor_t* seq_lens, const pa_tensor_t* query_start_loc,
                          int32_t max_query_len, float scale, float kv_scale, const pa_tensor_t* out,
                          const pa_tensor_t* lse, pa_stream_t stream);

int paged_attn_mla_decode_ex(const pa_tensor_t* q, const pa_tensor_t* kv_cache,
                             const pa_tensor_t* block_tables, const pa_tensor_t* seq_lens,
                             const pa_tensor_t* query_start_loc, int32_t max_query_len, float scale,
                             float kv_scale, const pa_tensor_t* out, const pa_tensor_t* lse,
                             const pa_options_t* opts, pa_stream_t stream);

/* Launch plan of paged_attn_mla_decode for a shape (kv_dtype: PA_BF16 or PA_FP8_E4M3);
 * opts may be NULL.  heads_per_cta reports the query heads of one chunk, row_tiles the
 * 16-row tiles of a chunk, num_ctas the split CTAs (each runs threads_per_cta threads in
 * one or two independent teams).  Reads device attributes only. */
int paged_attn_mla_plan(int32_t num_seqs, int32_t num_q_heads, int32_t kv_dtype, int32_t max_query_len,
                        const pa_options_t* opts, pa_plan_t* plan);

/* Bytes of split workspace an MLA call with this shape needs; paged_attn_mla_reserve grows
 * the library-owned workspace to fit it (call before capturing a CUDA graph). */
int paged_attn_mla_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t kv_dtype,
                                  int32_t max_query_len, size_t* bytes);
int paged_attn_mla_reserve(int32_t num_seqs, int32_t num_q_heads, int32_t kv_dtype, int32_t max_query_len);

/* Plan for a shape on the current device (kv_dtype: PA_BF16 or PA_FP8_E4M3).
 * opts may be NULL.  Reads device attributes only; enqueues nothing. */
int paged_attn_plan(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t kv_dtype, int32_t max_query_len, const pa_options_t* opts,
                    pa_plan_t* plan);

/* Bytes of split workspace a call with this shape needs (same as plan.workspace_bytes). */
int paged_attn_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t kv_dtype, int32_t max_query_len,
                              size_t* bytes);

/* Grow the library-owned workspace of the current device to fit this shape.  Call it
 * (or one ordinary decode call) before capturing paged_attn_decode in a CUDA graph:
 * during capture the library never allocates and returns PA_ERR_WORKSPACE instead.
 * Synchronises the device if it has to reallocate. */
int paged_attn_reserve(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                       int32_t kv_dtype, int32_t max_query_len);

/* Release the library-owned workspace of the current device (synchronises the device). */
int paged_attn_release(void);

/* Read the device status word of the current device into *flags (bit 0: page id out of
 * range; bit 1: seq_len < query length; bit 2: query length outside [1, max_query_len]
 * or query_start_loc inconsistent; bit 3: a pipeline wait timed out; bit 4: a query value
 * overflowed the f16 range on the fp8 path, or an MLA partial output did).  clear != 0 resets it to 0.  Synchronises
 * the device: a debugging aid, not for the hot path. */
int paged_attn_device_status(uint32_t* flags, int32_t clear);

/* Static description of a status code. */
const char* paged_attn_error_string(int status);

/* Detail of the last failing call on this thread ("" if none). */
const char* paged_attn_last_error_message(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t paged_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_ATTN_H */
