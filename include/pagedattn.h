/*
 * libpagedattn -- attention over a paged KV cache on one NVIDIA GB300 (sm_103a).
 *
 * Plain C ABI.  Every pointer argument is a DEVICE pointer unless it is
 * marked "host"; sizes are in elements unless marked "bytes".  "Device
 * pointer" means an address the kernels can access: device memory, or pinned
 * host memory mapped into the device's address space (cudaHostAlloc /
 * cudaHostRegister), which the kernels then read or write over the host link
 * -- for bf16 with head_dim 128, pa_decode and pa_decode_kv_write accept q
 * and out there, and pa_decode_kv_write also k_new / v_new (tested); the
 * caches, metadata and workspaces must be device memory.  The caller
 * owns every buffer (inputs, caches, outputs, workspace); the library
 * allocates no device memory.  Every call validates its arguments on the host
 * first: on a non-OK status nothing has been enqueued.  On PA_OK the work is
 * enqueued on `stream` and runs asynchronously; a later device-side problem
 * (an out-of-range page id or slot the host could not see) is never turned
 * into an out-of-bounds access -- the kernel skips the access and raises a
 * flag that pa_read_device_errors() returns.
 *
 * Cache layout (nano-vLLM learning note, allocate_kv_cache listing):
 *   k_cache, v_cache: [num_pages, page_size, num_kv_heads, head_dim], row-major.
 *   Flat slot s = page * page_size + offset holds one token's
 *   num_kv_heads * head_dim elements.
 * Query-head grouping (nano-vLLM learning note, Qwen3Attention.forward
 * listing): q-head h reads kv-head h / (num_q_heads / num_kv_heads).
 *
 * Padding rows: a request with context_lens[b] == 0 is padding (a batch
 * padded up to a fixed size, whose rows past the live requests keep the zero
 * lengths of buffers created zeroed: nano-vLLM learning note,
 * ModelRunner.capture_cudagraph listing).  Every call skips it silently: its
 * new tokens get position 0 and slot -1, nothing is read or stored for it,
 * its output rows are left untouched, and no PA_DEVERR_* flag is raised.
 * Negative lengths and lengths beyond the bounds stay errors.
 *
 * Supported: dtype fp32 or bf16; head_dim 64 or 128; num_kv_heads a power of
 * two <= 8; group size num_q_heads / num_kv_heads in 1..8; page_size a power
 * of two >= 16.  All vector pointers and row strides must be 16-byte aligned.
 *
 * Stream order: each call's first kernel starts after the stream's previous
 * work has completed.  The KV-write kernels (pa_kv_write and the two norm /
 * rotary writes) allow programmatically dependent kernels to launch at their
 * start (griddepcontrol.launch_dependents): a kernel the caller enqueues
 * after them with programmatic stream serialisation must wait
 * (griddepcontrol.wait, cudaGridDependencySynchronize) before it reads what
 * they write -- as the CUDA programming model asks of any such kernel.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

/* The library is built with hidden visibility; only these entry points are exported. */
#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_NULL = 1,        /* a required pointer is NULL */
  PA_ERR_DTYPE = 2,       /* dtype is neither PA_F32 nor PA_BF16 */
  PA_ERR_SHAPE = 3,       /* a count, size or stride is out of range */
  PA_ERR_ALIGN = 4,       /* a pointer or row stride is not 16-byte aligned */
  PA_ERR_UNSUPPORTED = 5, /* well-formed but outside the supported set */
  PA_ERR_WORKSPACE = 6,   /* workspace missing or smaller than required */
  PA_ERR_CUDA = 7,        /* a CUDA call or launch failed (pa_last_cuda_error) */
  PA_ERR_VALIDATION = 8,  /* reserved for callers of pa_validate_metadata */
  PA_ERR_CAPACITY = 9     /* block manager: not enough free blocks (or host memory) */
} pa_status;

typedef enum pa_dtype { PA_F32 = 0, PA_BF16 = 1 } pa_dtype;

/* Shape of one layer's cache and of the attention heads that read it. */
typedef struct pa_cache_desc {
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;
  int64_t num_pages;
  int32_t dtype; /* pa_dtype */
} pa_cache_desc;

/* A cudaStream_t passed as an opaque pointer; NULL is the legacy default stream. */
typedef void* pa_stream_t;

/* Device-side flags returned by pa_read_device_errors(). */
#define PA_DEVERR_BAD_SLOT 0x1u     /* a slot outside [-1, num_pages*page_size) was skipped */
#define PA_DEVERR_BAD_PAGE 0x2u     /* a block-table entry outside [0, num_pages) was skipped */
#define PA_DEVERR_BAD_LENGTH 0x4u   /* a context / chunk length was inconsistent; request skipped */
#define PA_DEVERR_TIMEOUT 0x8u      /* a bounded wait on an async copy gave up; output invalid */

/*
 * pa_slot_mapping -- positions and physical slots of each request's new tokens.
 *
 * Defined by the nano-vLLM learning note's prepare_prefill listing (new tokens
 * of a request sit at positions num_cached .. num_cached + num_new - 1) and
 * prepare_decode listing (slot = block_table[pos / page_size] * page_size +
 * pos % page_size).
 *
 *   batch            requests B (host).
 *   cu_seqlens_q     int32 [B+1], 0 = cu[0] <= cu[1] <= ... ; request b's new
 *                    tokens are rows cu[b] .. cu[b+1]-1 of the packed batch.
 *                    Decode is the case cu = 0, 1, ..., B.
 *   context_lens     int32 [B], tokens of request b INCLUDING its new ones.
 *   block_tables     int32 [B, max_pages_per_seq], physical page ids.
 *   num_tokens       cu[B] (host).
 *   positions        int32 [num_tokens] out: context_lens[b] - n_b + j.
 *   slot_mapping     int64 [num_tokens] out; -1 (and PA_DEVERR_* raised) for a
 *                    token whose page entry is out of range; -1 (no flag) for
 *                    the tokens of a padding row (context_lens[b] == 0).
 */
PA_API pa_status pa_slot_mapping(const pa_cache_desc* desc, int32_t batch, const int32_t* cu_seqlens_q,
                          const int32_t* context_lens, const int32_t* block_tables,
                          int32_t max_pages_per_seq, int64_t num_tokens, int32_t* positions,
                          int64_t* slot_mapping, pa_stream_t stream);

/*
 * pa_kv_write -- scatter each new token's K and V row into its cache slot.
 *
 * Defined by the nano-vLLM learning note's store_kvcache_kernel listing: row t
 * of k (v) is copied bit for bit to flat slot slot_mapping[t] of k_cache
 * (v_cache); slot -1 stores nothing.
 *
 *   k, v             [num_tokens, num_kv_heads, head_dim] rows, row t at
 *                    k + t * k_row_stride (elements, >= num_kv_heads*head_dim,
 *                    a multiple of 16 bytes).  May be views into a fused qkv.
 *   slot_mapping     int64 [num_tokens]; entries outside [-1, num_pages *
 *                    page_size) are skipped and flagged PA_DEVERR_BAD_SLOT.
 *   k_cache, v_cache caches as described at the top of this file.
 */
PA_API pa_status pa_kv_write(const pa_cache_desc* desc, const void* k, int64_t k_row_stride,
                      const void* v, int64_t v_row_stride, int64_t num_tokens,
                      const int64_t* slot_mapping, void* k_cache, void* v_cache,
                      pa_stream_t stream);

/*
 * pa_qk_norm_rope_kv_write -- per-head RMSNorm of q and k, rotary embedding of
 * both at absolute positions, then the KV write of (k, v).
 *
 * Defined by the nano-vLLM learning note: RMSNorm.rms_forward listing (mean of
 * squares in fp32, x * rsqrt(mean + eps) cast back to the dtype, then times
 * the weight), apply_rotary_emb and inv_freq listings (half-split rotation,
 * frequency theta^(-2i/head_dim), evaluated in fp32 and cast back), and the
 * Qwen3Attention.forward listing for the order (norm, rotary, store, attend).
 *
 *   q                [num_tokens, num_q_heads, head_dim] rows at q_row_stride.
 *   k, v             rows at k_row_stride / v_row_stride (as pa_kv_write).
 *   positions        int32 [num_tokens], absolute positions (pa_slot_mapping).
 *   q_norm_w, k_norm_w  [head_dim] weights in the cache dtype.
 *   eps, rope_theta  RMSNorm epsilon and rotary base (host).
 *   q_out            [num_tokens, num_q_heads, head_dim] contiguous output; it
 *                    may equal q only when q_row_stride == num_q_heads*head_dim.
 *   slot_mapping     as pa_kv_write; the normed, rotated k and the unchanged v
 *                    are written there.
 */
PA_API pa_status pa_qk_norm_rope_kv_write(const pa_cache_desc* desc, const void* q, int64_t q_row_stride,
                                   const void* k, int64_t k_row_stride, const void* v,
                                   int64_t v_row_stride, int64_t num_tokens,
                                   const int32_t* positions, const void* q_norm_w,
                                   const void* k_norm_w, float eps, float rope_theta,
                                   const int64_t* slot_mapping, void* q_out, void* k_cache,
                                   void* v_cache, pa_stream_t stream);

/*
 * pa_prefill_qk_norm_rope_kv_write -- pa_slot_mapping and
 * pa_qk_norm_rope_kv_write of a varlen prefill batch in one kernel: each new
 * token's position and cache slot are derived from the batch metadata as
 * pa_slot_mapping derives them (nano-vLLM learning note, prepare_prefill
 * listing), then its q and k are normed and rotated and (k, v) written.
 *
 *   q, k, v, q_norm_w, k_norm_w, eps, rope_theta, q_out, k_cache, v_cache
 *                    as pa_qk_norm_rope_kv_write.
 *   cu_seqlens_q, batch, context_lens, block_tables, max_pages_per_seq
 *                    as pa_slot_mapping (padding rows: position 0, slot -1).
 *   positions_out    optional int32 [num_tokens]: the positions (NULL: not written).
 *   slot_mapping_out optional int64 [num_tokens]: the slots (NULL: not written).
 * The cache, q_out and the optional outputs are those of pa_slot_mapping
 * followed by pa_qk_norm_rope_kv_write; the same metadata problems raise the
 * same device flags.
 */
PA_API pa_status pa_prefill_qk_norm_rope_kv_write(const pa_cache_desc* desc, const void* q, int64_t q_row_stride,
                                                  const void* k, int64_t k_row_stride, const void* v,
                                                  int64_t v_row_stride, int64_t num_tokens,
                                                  const int32_t* cu_seqlens_q, int32_t batch,
                                                  const int32_t* context_lens, const int32_t* block_tables,
                                                  int32_t max_pages_per_seq, const void* q_norm_w,
                                                  const void* k_norm_w, float eps, float rope_theta, void* q_out,
                                                  void* k_cache, void* v_cache, int32_t* positions_out,
                                                  int64_t* slot_mapping_out, pa_stream_t stream);

/*
 * pa_decode_workspace_size -- bytes of device workspace pa_decode needs for
 * these host-side sizes on the CURRENT device (the split plan depends on its SM
 * count).  max_ctas: 0 for the library's choice, else an upper bound on the
 * number of key-range partitions.  Returns 0 on an invalid descriptor or when no
 * CUDA device is usable.
 */
PA_API size_t pa_decode_workspace_size(const pa_cache_desc* desc, int32_t batch, int32_t max_context_len,
                                int32_t max_ctas);

/*
 * pa_decode_plan_info -- how pa_decode would split this batch on the CURRENT
 * device (host outs, either may be NULL): the number of key-range partitions
 * (CTAs; a merge kernel runs when it is above 1) and the tokens per chunk that
 * one pipeline stage moves.  Same arguments and failure cases as
 * pa_decode_workspace_size.
 */
PA_API pa_status pa_decode_plan_info(const pa_cache_desc* desc, int32_t batch, int32_t max_context_len,
                                     int32_t max_ctas, int32_t* num_partitions, int32_t* tokens_per_chunk);

/*
 * pa_decode -- batched GQA decode attention over the paged cache.
 *
 * For each request b and q-head h: out[b, h] = sum_j softmax_j(scale * q[b,h] .
 * K_j) V_j over the request's keys j < context_lens[b], found through
 * block_tables[b] (nano-vLLM learning note, Attention.forward listing: decode
 * attends to the cache after the step's KV write; prepare_decode listing:
 * context_lens counts the new token).
 *
 * The keys of all requests are cut into equal shares, one per CTA; a request
 * spread over several CTAs gets per-share (o, log-sum-exp) partials that a
 * second kernel merges (split-KV).  Shares depend only on context_lens, so the
 * result is bitwise independent of which physical pages hold the keys.  Up to
 * 512 requests every CTA computes the shares itself (the call launches the
 * decode kernel and, when some request is split, the merge kernel); beyond,
 * a one-CTA plan kernel computes them first.
 *
 *   q                [batch, num_q_heads, head_dim] contiguous.
 *   block_tables     int32 [batch, max_pages_per_seq].
 *   context_lens     int32 [batch], each in [1, max_context_len], or 0 for a
 *                    padding row (skipped silently, output untouched); a
 *                    request outside that range is skipped (its output
 *                    untouched) and flagged PA_DEVERR_BAD_LENGTH.
 *   max_context_len  host upper bound on context_lens (sizes the split plan).
 *   scale            softmax scale (host), e.g. 1/sqrt(head_dim).
 *   max_ctas         0 = library choice; else at most this many partitions
 *                    (1 = no split).
 *   out              [batch, num_q_heads, head_dim] contiguous, cache dtype.
 *   workspace        >= pa_decode_workspace_size(...) bytes, 256-byte aligned;
 *                    no initialisation needed; not shared with a concurrent call.
 */
PA_API pa_status pa_decode(const pa_cache_desc* desc, const void* q, int32_t batch, const void* k_cache,
                    const void* v_cache, const int32_t* block_tables, int32_t max_pages_per_seq,
                    const int32_t* context_lens, int32_t max_context_len, float scale,
                    int32_t max_ctas, void* out, void* workspace, size_t workspace_bytes,
                    pa_stream_t stream);

/*
 * pa_decode_kv_write -- the decode step's KV write and decode attention in one
 * launch sequence: for each request b, row b of k_new / v_new is stored into
 * the slot of position context_lens[b] - 1 (the slot pa_slot_mapping gives:
 * block_tables[b][pos / page_size] * page_size + pos % page_size) and the
 * request's query attends to its context_lens[b] keys, the new one included
 * (nano-vLLM learning note, Attention.forward: store the new K/V, then
 * attend).  Equal to pa_slot_mapping + pa_kv_write + pa_decode, bit for bit
 * in the cache and the output, without their two extra launches: the new row
 * is read straight from k_new / v_new and stored by the CTA that attends to it.
 *
 *   k_new, v_new     [batch, num_kv_heads, head_dim] rows at k_row_stride /
 *                    v_row_stride (elements, 16-byte multiples).
 *   slot_mapping     optional int64 [batch] out: the slot written for each
 *                    request, -1 for a padding row (context_lens[b] == 0:
 *                    nothing stored) or a request skipped for bad metadata.
 *   other arguments  as pa_decode; the workspace size is pa_decode's.
 * Needs num_pages * page_size < 2^31 (else PA_ERR_UNSUPPORTED).
 */
PA_API pa_status pa_decode_kv_write(const pa_cache_desc* desc, const void* q, const void* k_new,
                                    int64_t k_row_stride, const void* v_new, int64_t v_row_stride,
                                    int32_t batch, void* k_cache, void* v_cache, const int32_t* block_tables,
                                    int32_t max_pages_per_seq, const int32_t* context_lens,
                                    int32_t max_context_len, float scale, int32_t max_ctas,
                                    int64_t* slot_mapping, void* out, void* workspace,
                                    size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_decode_no_alloc -- pa_decode for callers that cannot allocate device
 * memory.  The pages have no counterpart of this call.
 *
 * For code that cannot call cudaMalloc where it runs decode (a plugin handed
 * only its buffers, a framework that forbids allocations at that point, a
 * process whose memory manager owns the device heap).  Arguments and
 * results are pa_decode's, without the workspace: the split-KV scratch comes
 * from a 16 MiB array inside the library that every device loading the
 * library holds until the process exits.  The call allocates nothing.
 *   - A batch whose plan needs more than 16 MiB of scratch (see
 *     pa_decode_workspace_size) is rejected with PA_ERR_WORKSPACE before
 *     anything is enqueued.
 *   - The first call on a device looks up the array's device address with a
 *     host-side runtime query (once per device).  With lazy module loading
 *     (CUDA_MODULE_LOADING=LAZY, the CUDA runtime's default) that lookup is
 *     also when the array is placed in the device's memory, so make the first
 *     call early -- before the caller's memory manager takes the rest of the
 *     heap, and before any stream capture.  Later calls allocate nothing.
 *   - Every call shares the array and it keeps the last call's contents;
 *     nothing in it has to start at zero, but calls that overlap on the GPU
 *     (two streams, two host threads) race on it.
 */
PA_API pa_status pa_decode_no_alloc(const pa_cache_desc* desc, const void* q, int32_t batch,
                                    const void* k_cache, const void* v_cache, const int32_t* block_tables,
                                    int32_t max_pages_per_seq, const int32_t* context_lens,
                                    int32_t max_context_len, float scale, int32_t max_ctas, void* out,
                                    pa_stream_t stream);

/*
 * pa_prefill_varlen -- chunked-prefill attention for packed new tokens.
 *
 * Request b's chunk is rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 of q (flat
 * varlen packing, qwen-engine README); those n_b tokens are the last n_b of its
 * context_lens[b] tokens, so row i sits at position context_lens[b] - n_b + i
 * and attends to keys 0 .. that position: the cached prefix plus the causal
 * part of its own chunk, all read from the cache (nano-vLLM learning note,
 * Attention.forward listing: with block tables, k and v come from the cache
 * after the step's KV write).
 *
 *   q                [num_tokens, num_q_heads, head_dim] contiguous (already
 *                    normed and rotated, e.g. q_out of pa_qk_norm_rope_kv_write).
 *   cu_seqlens_q     int32 [batch+1] as in pa_slot_mapping; num_tokens = cu[batch].
 *   max_seqlen_q     host upper bound on n_b.
 *   context_lens     int32 [batch], n_b <= context_lens[b] <= max_context_len,
 *                    or 0 for a padding row (its rows of out are untouched).
 *   scale            softmax scale (host), finite and > 0.
 *   out              [num_tokens, num_q_heads, head_dim] contiguous.
 * bf16 with head_dim 128 runs on the tcgen05 tensor cores; other cases on a
 * CUDA-core kernel.
 *   workspace        optional device buffer (256-byte aligned) of
 *                    workspace_bytes >= pa_prefill_workspace_size(...), used
 *                    only by the tensor-core path; owned by the caller, not
 *                    read by the host, contents need not be initialised.  With
 *                    it, a planner kernel splits long key ranges over several
 *                    CTAs and orders the work longest first, and a merge
 *                    kernel combines the parts by their log-sum-exp (the
 *                    decode split-KV rule); without it
 *                    (NULL) each CTA takes one pair of 128-row q-tiles with
 *                    all its keys.  Results
 *                    agree within the bf16 tolerance either way; a too small
 *                    workspace returns PA_ERR_WORKSPACE.  Calls sharing one
 *                    workspace must be ordered on the GPU (same stream).
 *                    Once a planned call has run, the workspace's first 16
 *                    bytes hold int32 {CTAs per kv-head, split pairs, part
 *                    size in 128-key tiles, q-tile pairs} (diagnostics).
 */
PA_API pa_status pa_prefill_varlen(const pa_cache_desc* desc, const void* q, const int32_t* cu_seqlens_q,
                                   int32_t batch, int32_t max_seqlen_q, int64_t num_tokens, const void* k_cache,
                                   const void* v_cache, const int32_t* block_tables, int32_t max_pages_per_seq,
                                   const int32_t* context_lens, int32_t max_context_len, float scale, void* out,
                                   void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_prefill_step -- one chunked-prefill step in one call: the step's KV write
 * (nano-vLLM learning note, Attention.forward listing: store_kvcache before
 * the attention), then pa_prefill_varlen over the cache.
 *
 * With q_norm_w and k_norm_w: pa_prefill_qk_norm_rope_kv_write (q normed and
 * rotated into q_out, positions_out and slot_mapping_out optional), then
 * pa_prefill_varlen on q_out.  With both NULL: pa_slot_mapping into
 * positions_out and slot_mapping_out (both required), pa_kv_write of k and v,
 * then pa_prefill_varlen on q itself (q_row_stride must then be
 * num_q_heads*head_dim; q_out, eps and rope_theta are unused).  One NULL
 * weight is PA_ERR_NULL.
 *
 * Every argument has the meaning, layout and ownership it has in those calls;
 * all of them are checked before anything is enqueued.  The cache, q_out,
 * positions_out, slot_mapping_out and out are exactly those of the calls made
 * one after another.  The difference is the launch: the attention planner
 * (workspace given, bf16 with head_dim 128) reads only cu_seqlens_q and
 * context_lens, which the write kernel does not write, so here it runs beside
 * that kernel instead of after it (programmatic dependent launch; the
 * attention kernel still starts on the cache only once the write is
 * complete).  pa_prefill_varlen alone cannot know which kernel wrote its
 * metadata, so its planner starts only after the previous kernel completes.
 */
PA_API pa_status pa_prefill_step(const pa_cache_desc* desc, const void* q, int64_t q_row_stride, const void* k,
                                 int64_t k_row_stride, const void* v, int64_t v_row_stride, int64_t num_tokens,
                                 const int32_t* cu_seqlens_q, int32_t batch, int32_t max_seqlen_q,
                                 const int32_t* context_lens, int32_t max_context_len, const int32_t* block_tables,
                                 int32_t max_pages_per_seq, const void* q_norm_w, const void* k_norm_w, float eps,
                                 float rope_theta, float scale, void* q_out, void* k_cache, void* v_cache,
                                 int32_t* positions_out, int64_t* slot_mapping_out, void* out, void* workspace,
                                 size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_prefill_workspace_size -- bytes of the optional pa_prefill_varlen
 * workspace for these bounds on the current device (it holds the work list
 * and, for split ranges, fp32 partial outputs of at most 4 waves of CTAs:
 * about 80 MiB on a 152-SM GPU), or 0 when the call would not use one
 * (fp32 or head_dim 64, max_context_len beyond 65535 * 128) or the
 * arguments are invalid.
 */
PA_API size_t pa_prefill_workspace_size(const pa_cache_desc* desc, int32_t batch, int32_t max_seqlen_q,
                                        int64_t num_tokens, int32_t max_context_len);

/*
 * pa_validate_metadata -- opt-in device check of the metadata the other calls
 * trust.  Counts, into *error_count (device int32, overwritten), the requests
 * with context_lens outside [1, min(max_context_len, max_pages_per_seq *
 * page_size)] (padding rows, context_lens == 0, are not counted), new-token counts that are negative or exceed the context (when
 * cu_seqlens_q is given; may be NULL), and block-table entries outside
 * [0, num_pages) among the pages a request uses.  Never faults; read the count
 * after synchronising.
 */
PA_API pa_status pa_validate_metadata(const pa_cache_desc* desc, int32_t batch,
                               const int32_t* cu_seqlens_q, const int32_t* context_lens,
                               const int32_t* block_tables, int32_t max_pages_per_seq,
                               int32_t max_context_len, int32_t* error_count, pa_stream_t stream);

/*
 * pa_selftest_bounded_wait -- exercises the kernels' bounded-wait path.  Launches
 * one thread that waits on an mbarrier nothing ever arrives on; after
 * timeout_ms (1 .. 10000) the wait gives up, the kernel raises
 * PA_DEVERR_TIMEOUT and exits, and the context stays usable.  Every wait in
 * the other kernels ends the same way (with a 2 s limit), so a lost copy or
 * MMA completion costs a flagged, wrong result instead of a hung GPU.
 */
PA_API pa_status pa_selftest_bounded_wait(int32_t timeout_ms, pa_stream_t stream);

/*
 * pa_read_device_errors -- the PA_DEVERR_* flags raised on the current device
 * since the last reset (host out).  Synchronises the device.  reset != 0
 * clears the flags.
 */
PA_API pa_status pa_read_device_errors(uint32_t* flags, int32_t reset);

/* CUDA error code behind the calling thread's last PA_ERR_CUDA (0 if none). */
PA_API int32_t pa_last_cuda_error(void);

/* Static description of a status code. */
PA_API const char* pa_status_string(pa_status status);

/* ---------------------------------------------------------------------------
 * Host block manager (nano-vLLM learning note: Block, BlockManager,
 * compute_hash, can_allocate, allocate, deallocate, can_append, may_append and
 * hash_blocks listings).  Decides which physical page (block) holds each
 * token of each sequence and shares full pages between sequences whose
 * prompts start with the same tokens (prefix caching): every full block that
 * has been computed is registered under a hash of its tokens chained with the
 * previous block's hash, and a new sequence reuses its leading registered
 * blocks (never its last block) whose stored tokens match.  Free blocks are a
 * FIFO: allocation takes the oldest, a released block goes to the back and
 * keeps its hash until it is handed out again.  Host memory only: the outputs
 * (block tables, context lengths, slots) are host arrays the caller uploads.
 * A manager is not thread-safe.  Sequences are named by caller-chosen int64
 * ids.  The hash is a chained SplitMix64 mix of the 32-bit token ids (the
 * pages use xxHash64); hits are confirmed by comparing tokens.
 * ------------------------------------------------------------------------- */
typedef struct pa_block_manager pa_block_manager;

/* A manager of num_blocks blocks of block_size tokens, all free.  *out is set
 * to NULL on error.  PA_ERR_CAPACITY if host memory runs out. */
PA_API pa_status pa_bm_create(int64_t num_blocks, int32_t block_size, pa_block_manager** out);
PA_API void pa_bm_destroy(pa_block_manager* m);

/* How many leading blocks of a prompt of num_tokens token ids (host) would be
 * reused from the cache, or -1 in *num_cached_blocks when the free blocks do
 * not cover the rest.  Changes nothing. */
PA_API pa_status pa_bm_can_allocate(pa_block_manager* m, const int32_t* token_ids, int64_t num_tokens,
                                    int64_t* num_cached_blocks);

/* Register sequence seq_id with its prompt and give it ceil(num_tokens /
 * block_size) blocks, the leading cached ones shared.  *num_cached_tokens
 * (optional) = tokens whose K/V are already in the shared blocks (a multiple
 * of block_size): the caller computes and writes only the rest.
 * PA_ERR_CAPACITY (nothing changed) when the free blocks do not suffice;
 * PA_ERR_SHAPE when seq_id is already registered. */
PA_API pa_status pa_bm_allocate(pa_block_manager* m, int64_t seq_id, const int32_t* token_ids, int64_t num_tokens,
                                int64_t* num_cached_tokens);

/* Append one token (decode); a sequence whose length becomes 1 mod
 * block_size gets a fresh block.  PA_ERR_CAPACITY (nothing changed) when that
 * block is not available. */
PA_API pa_status pa_bm_append_token(pa_block_manager* m, int64_t seq_id, int32_t token_id);

/* Declare the first num_computed_tokens tokens of seq_id computed (their K/V
 * written): its full blocks among them are registered for prefix reuse. */
PA_API pa_status pa_bm_hash_blocks(pa_block_manager* m, int64_t seq_id, int64_t num_computed_tokens);

/* Release seq_id: one reference less on each of its blocks, last block first;
 * blocks nobody holds go to the back of the free list. */
PA_API pa_status pa_bm_free(pa_block_manager* m, int64_t seq_id);

/* Host int32 block_tables [num_seqs, max_pages_per_seq] for these sequences
 * (unused entries = pad_page, e.g. a reserved page), and optionally their
 * lengths in context_lens [num_seqs].  PA_ERR_SHAPE (nothing written) for an
 * unknown id or a table longer than max_pages_per_seq. */
PA_API pa_status pa_bm_block_tables(pa_block_manager* m, const int64_t* seq_ids, int32_t num_seqs,
                                    int32_t max_pages_per_seq, int32_t pad_page, int32_t* block_tables,
                                    int32_t* context_lens);

/* Host int64 slots of the last num_new_tokens[i] tokens of each sequence, in
 * order (sum(num_new_tokens) entries): block * block_size + offset, the
 * values pa_slot_mapping computes on the device. */
PA_API pa_status pa_bm_slot_mapping(pa_block_manager* m, const int64_t* seq_ids, int32_t num_seqs,
                                    const int32_t* num_new_tokens, int64_t* slot_mapping);

/* Counters (each output optional). */
PA_API pa_status pa_bm_query(pa_block_manager* m, int64_t* num_free_blocks, int64_t* num_seqs,
                             int64_t* num_hashed_blocks);
PA_API pa_status pa_bm_block_ref_count(pa_block_manager* m, int32_t block_id, int32_t* ref_count);
PA_API pa_status pa_bm_seq_info(pa_block_manager* m, int64_t seq_id, int64_t* num_tokens,
                                int64_t* num_cached_tokens, int32_t* num_blocks);

/* Library version, major * 10000 + minor * 100 + patch. */
PA_API int32_t pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
