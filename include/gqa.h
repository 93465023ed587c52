/*
 * gqa.h -- C ABI of libgqa: GroupQueryAttention over a shared, pre-allocated
 * BNSH key/value buffer, for one NVIDIA GB300 (sm_103a).
 *
 * What one call computes (sources: the onnxruntime discussion "Clarification
 * about GroupQueryAttention behavior" -- the quoted past_key text and
 * tianleiwu's reply; the torch-mlir PR "[TorchOnnxToTorch] Add pad+scatter KV
 * cache and mask to GQA" -- its description; the rocMLIR discussion "KV
 * Cache" -- "Example" and "Short summary of notes"):
 *
 *   for every sequence b with past length P_b = seqlens_k[b] and every new
 *   token i < S, at position p = P_b + i:
 *   (1) rotary embedding of the new query and key rows at position p
 *       (position ids = arange plus the past length);
 *   (2) the rotated key row and the value row are written into the shared
 *       buffer at slot p of every KV head (scatter-append at seqlens_k);
 *   (3) query head h attends over KV head h / (H / Hkv), over keys
 *       j <= p (causal) and, when local_window_size W > 0, j > p - W; the
 *       scan stops at the sequence's true length P_b + S, never at
 *       max_seq_len; an optional additive attention_bias is added to the
 *       scaled scores;
 *   (4) when the buffer has no room for the new tokens the call fails with
 *       GQA_ERR_KV_OVERFLOW and writes nothing -- unless the caller selects
 *       the sliding-window cache (dims->kv_eviction = 1; the SWA follow-up of
 *       the onnxruntime discussion: the op keeps only the
 *       min(total_sequence_length, cache_capacity) most recent tokens,
 *       contiguously), in which case the oldest tokens make way.
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" are CUDA device pointers on the current
 *     device; "host" pointers are ordinary host memory.  All device pointers
 *     must be 16-byte aligned.
 *   - The caller owns every buffer.  The library allocates no device memory
 *     per call; it keeps one small error word per device in a static device
 *     variable.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream).  Argument errors and overflow that the host can see
 *     are reported before anything is launched, so no buffer is touched.
 *     Errors only the device can see (a seqlens_k entry beyond the buffer, a
 *     bounded wait inside a kernel that ran out) are recorded in the device
 *     error word; the kernels skip the affected writes and never trap.
 *     gqa_check_device_status() reports and clears that word.
 *   - No function throws across the ABI.
 */
#ifndef GQA_H_
#define GQA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GQA_OK = 0,
  GQA_ERR_INVALID_ARGUMENT = 1, /* bad dims, null or misaligned pointer, small workspace */
  GQA_ERR_KV_OVERFLOW = 2,      /* the shared buffer has no room for the new tokens */
  GQA_ERR_UNSUPPORTED = 3,      /* a valid operator form this library does not implement */
  GQA_ERR_CUDA = 4,             /* a CUDA runtime call failed */
  GQA_ERR_TIMEOUT = 5           /* a bounded wait inside a kernel ran out */
} gqa_status_t;

typedef enum { GQA_DTYPE_FP16 = 0, GQA_DTYPE_BF16 = 1 } gqa_dtype_t;

/* Problem dimensions.  All are runtime values. */
typedef struct {
  int32_t batch;              /* B >= 1 */
  int32_t seq_len;            /* S >= 1: new tokens per sequence (1 = decode) */
  int32_t num_heads;          /* H: query heads */
  int32_t kv_num_heads;       /* Hkv: key/value heads; H % Hkv == 0 */
  int32_t head_size;          /* D: multiple of 8, at most 256 */
  int32_t max_seq_len;        /* M: slots per (sequence, KV head) in the shared buffer */
  int32_t dtype;              /* gqa_dtype_t: element type T of every T array */
  int32_t rotary_interleaved; /* 0: dimension j pairs with j + D/2; 1: j pairs with j + 1 (2j, 2j+1) */
  int32_t cos_cache_rows;     /* rows of cos/sin caches; ignored when cos_cache is NULL */
  int32_t bias_batch;         /* 1 or B; ignored when attention_bias is NULL */
  int32_t bias_heads;         /* 1 or H; ignored when attention_bias is NULL */
  int32_t past_seq_len;       /* Mp: slots of past_key/past_value, 0 <= Mp <= M; read only
                                 when past_key is not present_key (non-shared binding) */
  int32_t kv_eviction;        /* 0: a full buffer is GQA_ERR_KV_OVERFLOW.  1: sliding-window
                                 cache of capacity M with contiguous eviction (shared binding
                                 only; see gqa_forward) */
} gqa_dims_t;

/*
 * gqa_forward -- one GroupQueryAttention step over the shared buffer.
 *
 *   dims             host: problem dimensions (above).
 *   query            device, T [B, S, H*D]   new query rows (heads contiguous per token).
 *                    Packed QKV (key and value both NULL): T [B, S, (H + 2 Hkv)*D], each
 *                    token's row holding its H query heads, then its Hkv key heads, then
 *                    its Hkv value heads, each head D contiguous elements (the
 *                    [batch, seq, hidden] -> [batch, seq, heads, head_size] reading of
 *                    "[TorchOnnxToTorch] Add pad+scatter KV cache and mask to GQA").
 *   key, value       device, T [B, S, Hkv*D] new key/value rows, or both NULL (packed).
 *                    Only one of them NULL is GQA_ERR_INVALID_ARGUMENT.
 *   past_key         device, T.  Two bindings ("Clarification about GroupQueryAttention
 *   present_key      behavior": the quoted past_key text and ZackyLake's summary):
 *   past_value       - shared: past_key == present_key and past_value == present_value,
 *   present_value      one buffer [B, Hkv, M, D] of max_sequence_length slots.  Only
 *                      slots [P_b, P_b + S) of each (b, KV head) are written; every
 *                      other slot keeps its bits.
 *                    - non-shared: four distinct, non-overlapping buffers (only
 *                      pointer equality is checked), past [B, Hkv, Mp, D]
 *                      (Mp = dims->past_seq_len) and present [B, Hkv, M, D].  The
 *                      present becomes past + new: slots [0, P_b) are copied from the
 *                      past, slots [P_b, P_b + S) get the new rows, later slots keep
 *                      their bits, and attention runs over the present.  The past is
 *                      not written.  A sequence with P_b > Mp records
 *                      GQA_ERR_INVALID_ARGUMENT on the device; its present slots below
 *                      P_b are not copied.
 *                    Only one of the two pairs equal (or a past buffer equal to the
 *                    other present buffer) returns GQA_ERR_INVALID_ARGUMENT.
 *   seqlens_k        device, int32 [B]: past length P_b of each sequence (0 = empty).
 *                    With kv_eviction = 1, P_b counts every earlier token of the
 *                    sequence (the absolute position of its first new token) and may
 *                    exceed M; the buffer then holds the min(P_b, M) most recent of
 *                    them at slots [0, min(P_b, M)), slot s holding position
 *                    P_b - min(P_b, M) + s.  After the call it holds the
 *                    min(P_b + S, M) most recent tokens the same way (slots beyond keep
 *                    their bits).  Token i attends over the cached tokens and the new
 *                    ones (positions P_b - min(P_b, M) ... P_b + i), with the causal
 *                    mask and window on absolute positions; rotary positions are
 *                    absolute.  A full buffer is then never an error; P_b < 0 or
 *                    P_b + S > total_sequence_length stays one (device-recorded
 *                    GQA_ERR_INVALID_ARGUMENT).  kv_eviction = 1 with the non-shared
 *                    binding returns GQA_ERR_UNSUPPORTED.
 *   total_sequence_length  host scalar: an upper bound on P_b + S for every b and the
 *                    last dimension of attention_bias.  Must be >= S.  Larger than M:
 *                    GQA_ERR_KV_OVERFLOW before any launch (allowed with
 *                    kv_eviction = 1).  A sequence with
 *                    P_b + S > M (or P_b < 0, or P_b + S > total_sequence_length) is
 *                    detected on the device: that sequence is skipped entirely (no
 *                    slot, no output row written) and the device error word records
 *                    GQA_ERR_KV_OVERFLOW (resp. GQA_ERR_INVALID_ARGUMENT).
 *   cos_cache,       device, T [cos_cache_rows, D/2]: cos/sin of the rotary angle of
 *   sin_cache        position p and pair j.  Both NULL: no rotary embedding.
 *                    cos_cache_rows must be >= total_sequence_length.
 *   scale            score scale; <= 0 means 1/sqrt(D).
 *   local_window_size  <= 0: full causal attention; W > 0: each token sees the W most
 *                    recent positions up to and including its own.
 *   attention_bias   device, T [bias_batch, bias_heads, S, total_sequence_length] or
 *                    NULL; indexed by absolute key position.
 *   output           device, T [B, S, H*D].
 *   workspace        device scratch of at least gqa_workspace_size() bytes (may be NULL
 *                    when that size is 0).  Its contents on entry do not matter.
 *   stream           cudaStream_t.
 *
 * Returns GQA_OK once the work is enqueued.
 */
gqa_status_t gqa_forward(const gqa_dims_t* dims,
                         const void* query, const void* key, const void* value,
                         const void* past_key, const void* past_value,
                         void* present_key, void* present_value,
                         const int32_t* seqlens_k, int32_t total_sequence_length,
                         const void* cos_cache, const void* sin_cache,
                         float scale, int32_t local_window_size,
                         const void* attention_bias,
                         void* output,
                         void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * gqa_workspace_size -- bytes of device scratch gqa_forward needs for these
 * dims, total_sequence_length and local_window_size: rotated queries for the
 * generic kernel (head sizes other than 128), key-range partials for a
 * tensor-core prefill grid of fewer than two CTAs per SM, split-KV partials
 * with their counters for decode, and with kv_eviction = 1 and
 * total_sequence_length > max_seq_len (a call that may evict) the rotated
 * queries and new key rows of the evicting path.  The figure is for the current
 * device and covers calls with or without rotary embedding and either
 * binding.  Returns 0 for invalid dims (and when no scratch is needed).
 */
size_t gqa_workspace_size(const gqa_dims_t* dims, int32_t total_sequence_length, int32_t local_window_size);

/*
 * gqa_check_device_status -- synchronise `stream`, then report and clear the
 * current device's error word (GQA_OK when no kernel recorded an error), or
 * GQA_ERR_CUDA when a CUDA call or an earlier launch failed.
 */
gqa_status_t gqa_check_device_status(void* stream);

/* gqa_status_string -- a static, human-readable name for a status code. */
const char* gqa_status_string(gqa_status_t status);

/*
 * gqa_decode_noalloc -- the decode step of gqa_forward (seq_len == 1,
 * head_size == 128, at most 16 query heads per KV head) without a workspace
 * argument.  The operator's pages have no counterpart to this entry point; it
 * exists for callers that cannot allocate device memory when they run the
 * step and have no scratch to pass -- for example an inference runtime whose
 * memory planner hands out every buffer ahead of execution, or a serving
 * loop in which cudaMalloc/cudaFree (which may synchronise the device) are
 * not allowed.
 *
 * Arguments, layouts and error behaviour are those of gqa_forward, minus
 * workspace/workspace_bytes.  The split-KV partial results go to a static
 * device array of 4 MiB inside the library (held by every GPU that loads it,
 * until exit; a 152-SM GB300 needs at most about 2.5 MB of it); a call that
 * would need more returns GQA_ERR_UNSUPPORTED before any launch, as do shapes
 * other than the decode shape above, the non-shared binding (separate past
 * and present buffers), packed QKV and kv_eviction = 1.  The function
 * allocates nothing.
 *   - All calls on one device share that array and it keeps the last call's
 *     contents (nothing in it needs to start at zero).  Calls whose kernels
 *     can overlap on the GPU race on it: order them on one stream.
 *   - The first call on each device looks up the array's device address
 *     with that device current; make that first call before any stream
 *     capture begins.
 */
gqa_status_t gqa_decode_noalloc(const gqa_dims_t* dims,
                                const void* query, const void* key, const void* value,
                                const void* past_key, const void* past_value,
                                void* present_key, void* present_value,
                                const int32_t* seqlens_k, int32_t total_sequence_length,
                                const void* cos_cache, const void* sin_cache,
                                float scale, int32_t local_window_size,
                                const void* attention_bias,
                                void* output,
                                void* stream);

/*
 * gqa_forward_host -- gqa_forward with the step's per-call inputs and its
 * output in page-locked HOST memory, for a caller whose step data lives on
 * the host while the shared buffer stays resident on the device.
 *
 *   query, key, value, seqlens_k, output
 *                    host, page-locked (cudaHostAlloc/cudaMallocHost, or
 *                    cudaHostRegister), same types and layouts as in
 *                    gqa_forward; query, key, value and output 16-byte
 *                    aligned, seqlens_k 4-byte aligned.  Any other pointer
 *                    (pageable or device memory) returns
 *                    GQA_ERR_INVALID_ARGUMENT before any launch.
 *   past_key, past_value, present_key, present_value, cos_cache, sin_cache,
 *   attention_bias   device, as in gqa_forward.
 *   workspace        device scratch of at least gqa_workspace_size_host()
 *                    bytes: gqa_forward's scratch plus device copies of the
 *                    step's inputs and output.
 *
 * The call enqueues three stages on `stream`: a copy kernel that reads the
 * inputs from host memory into the workspace, gqa_forward's kernels on those
 * copies, and a copy kernel that writes the output to host memory.  On the
 * decode path (seq_len 1, head_size 128, at most 16 query heads per KV head)
 * the attention kernel stores the output rows straight into the host output
 * and the last stage is not needed.  The output is valid once the stream
 * reaches the end of the call (e.g. after cudaStreamSynchronize).  The caller must not change the host inputs, or
 * read the host output, before then.  Error behaviour is gqa_forward's.
 */
gqa_status_t gqa_forward_host(const gqa_dims_t* dims,
                              const void* query, const void* key, const void* value,
                              const void* past_key, const void* past_value,
                              void* present_key, void* present_value,
                              const int32_t* seqlens_k, int32_t total_sequence_length,
                              const void* cos_cache, const void* sin_cache,
                              float scale, int32_t local_window_size,
                              const void* attention_bias,
                              void* output,
                              void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * gqa_workspace_size_host -- bytes of device scratch gqa_forward_host needs
 * (gqa_workspace_size() rounded up to 256, plus the staged query, key,
 * value, seqlens_k and output, each rounded up to 256).  0 for invalid dims.
 */
size_t gqa_workspace_size_host(const gqa_dims_t* dims, int32_t total_sequence_length,
                               int32_t local_window_size);

#ifdef __cplusplus
}
#endif

#endif /* GQA_H_ */
