/*
 * sinkattn: grouped-query attention with learned per-head sinks, for NVIDIA
 * GB300 (sm_103a). C ABI of libsinkattn.so.
 *
 * The operation. Page "GPT-OSS on day 0", section "Attention: GQA with
 * Attention Sinks": several query heads share one KV head, and every query
 * head owns one trained sink parameter that takes part in the softmax.
 * Section "Kernels for GPT-OSS / Sink Attention": the sink is one extra logit
 * beside the scaled Q.K products; it has no value row. For query row i of
 * sequence b and query head h (KV head g = h / (hq / hkv)):
 *
 *   p   = (Lk_b - Lq_b) + i          query position; queries are the last
 *                                     Lq_b of the Lk_b positions
 *   J   = { j < Lk_b : (!causal || j <= p) && (window == 0 || j > p - window) }
 *   s_j = scale * <q[i,h,:], k[j,g,:]>
 *   out = sum_{j in J} e^{s_j} v[j,g,:] / (e^{sink_h} + sum_{j in J} e^{s_j})
 *   lse = ln(e^{sink_h} + sum_{j in J} e^{s_j})
 *
 * The sink is not multiplied by `scale`. With sinks == NULL the sink term is
 * absent. A row with an empty J gets out = 0 and lse = sink_h (or -inf with no
 * sinks); it never produces NaN.
 *
 * The same section describes the online softmax (running maximum m and running
 * denominator d) and how the sink enters it: m starts at the head's sink
 * instead of -inf, with d = 1, and when the KV sequence is split into blocks
 * the sink enters exactly one block. The kernels behind this header do that.
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller, row-major,
 *    contiguous, 16-byte aligned. bf16 data is passed as `const void*`.
 *    Prefill outputs (out) and backward gradients (dq, dk, dv) that start on
 *    a 32-byte boundary are written with 32-byte stores, a faster path with
 *    bitwise the same results.
 *  - The library allocates no device memory and never synchronises: every
 *    call only enqueues work on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and returns. Device-side metadata (sequence offsets,
 *    lengths, block tables) is never read by the host, so calls can be
 *    captured in a CUDA graph.
 *  - Host-side argument errors return before anything is enqueued. A failed
 *    launch returns SINKATTN_ERR_CUDA. No C++ exception crosses the ABI.
 *  - head_dim must be 64 or 128 (SINKATTN_ERR_UNSUPPORTED otherwise; the
 *    backward takes 64 only) and hq must be a multiple of hkv. Below, D
 *    stands for head_dim.
 *  - Outputs: `out` is bf16 (round to nearest even) with the query layout;
 *    `lse` is float32, natural log, sink included; `lse` may be NULL.
 *  - Inputs must be finite. Rows of K/V outside a sequence may be read but get
 *    zero weight.
 */
#ifndef SINKATTN_H
#define SINKATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SINKATTN_OK = 0,
  SINKATTN_ERR_INVALID_ARGUMENT = 1, /* null/misaligned pointer, bad size */
  SINKATTN_ERR_UNSUPPORTED = 2,      /* valid but not implemented (head_dim != 64, ...) */
  SINKATTN_ERR_WORKSPACE_TOO_SMALL = 3,
  SINKATTN_ERR_CUDA = 4              /* a CUDA runtime/driver call failed */
} sinkattn_status_t;

/* Mask of one call. The pages do not describe windows; this library reads a
 * window of W as "the W most recent positions up to and including p". */
typedef struct {
  int causal;  /* nonzero: key j visible only if j <= p */
  int window;  /* 0: no window; W > 0: key j visible only if j > p - W */
  float scale; /* multiplies q.k; must be finite and > 0 */
} sinkattn_mask_t;

/* Human-readable name of a status code (static storage). */
const char *sinkattn_status_string(sinkattn_status_t status);

/* Name of the CUDA error behind the calling thread's most recent
 * SINKATTN_ERR_CUDA (e.g. "cudaErrorLaunchOutOfResources"), or "no CUDA
 * error"; static storage. */
const char *sinkattn_last_cuda_error(void);

/*
 * Prefill over packed variable-length sequences (page "Fast embeddings on
 * GPUs", section "ROSE": attention over ragged inputs without padding).
 *
 *   q        bf16 [total_q, hq, D]    sequence b owns rows cu_seqlens_q[b]..[b+1]
 *   k, v     bf16 [total_k, hkv, D]   sequence b owns rows cu_seqlens_k[b]..[b+1]
 *   cu_seqlens_q, cu_seqlens_k  int32 [batch+1], device, non-decreasing,
 *            starting at 0; the last entries equal total_q and total_k.
 *   total_q, total_k            host copies of those last entries (bounds for
 *            the tensor maps that stage Q/K/V tiles).
 *   max_seqlen_q, max_seqlen_k  host upper bounds on any sequence's length
 *            (grid sizing). A query length above max_seqlen_q is cut to the
 *            bound (the rows past it are not written) and recorded as code 3
 *            in the device error word.
 *   sinks    float32 [hq] or NULL.
 *   num_splits     key-range splits (section "Kernels for GPT-OSS / Sink
 *            Attention": the KV sequence split into blocks, the sink in one
 *            block only). 1 = none; n > 1 = every (query tile, head) item is
 *            cut into n key ranges, each writing a normalised partial output
 *            and lse (the first range alone starting from the sink), which a
 *            log-sum-exp merge then combines; at most 64. 0 = automatic: splits
 *            only when the call has too few (query tile, head) items to fill
 *            the GPU's SMs and long key ranges (e.g. a few hundred new tokens
 *            over a long context); the choice depends on the current device's
 *            SM count.
 *   out      bf16 [total_q, hq, D];    lse  float32 [total_q, hq] or NULL.
 *   workspace/workspace_bytes   device scratch, 256-byte aligned, at least
 *            sinkattn_prefill_workspace_size() bytes for the same arguments;
 *            contents need not be initialised. It receives an fp16 copy of v
 *            for the P.V product (values of magnitude above 65504 are clamped
 *            to +-65504 there), the list of query tiles that the persistent
 *            kernel works through, longest first, and with splits the fp32
 *            partials (splits * total_q * hq * (4 D + 4) bytes).
 * A sequence with Lq_b > Lk_b is allowed: its first Lq_b - Lk_b queries see no
 * key under a causal mask.
 */
size_t sinkattn_prefill_workspace_size(int batch, int64_t total_q, int64_t total_k,
                                       int max_seqlen_q, int max_seqlen_k, int hq, int hkv,
                                       int head_dim, int window, int num_splits);

sinkattn_status_t sinkattn_prefill(const void *q, const void *k, const void *v,
                                   const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                   int batch, int64_t total_q, int64_t total_k,
                                   int max_seqlen_q, int max_seqlen_k, int hq, int hkv,
                                   int head_dim, const float *sinks, sinkattn_mask_t mask,
                                   int num_splits, void *out, float *lse, void *workspace,
                                   size_t workspace_bytes, void *stream);

/*
 * Prefill over a paged KV cache: chunked prefill of new query tokens against
 * keys and values that live in fixed-size pages (page "Fast embeddings on
 * GPUs", section "ROSE": paged KV for serving; ragged sequences without
 * padding). Same operation, mask and outputs as sinkattn_prefill; only the
 * key/value addressing differs.
 *
 *   q        bf16 [total_q, hq, D]    sequence b owns rows cu_seqlens_q[b]..[b+1]
 *   cu_seqlens_q  int32 [batch+1], device, non-decreasing, starting at 0,
 *            last entry total_q.
 *   k_cache, v_cache  bf16 [num_pages, hkv, page_size, D]. Key j of sequence
 *            b is slot j % page_size of page block_table[b][j / page_size].
 *   block_table   int32 [batch, max_pages_per_seq], device.
 *   seqlens_k     int32 [batch], device: Lk_b, which counts the cached keys and
 *            the new tokens' own keys (already written into the pages). The
 *            queries are the last Lq_b of the Lk_b positions.
 *   max_seqlen_q  host upper bound on Lq_b (grid sizing).
 *   max_seqlen_k  host upper bound on Lk_b; must not exceed
 *            max_pages_per_seq * page_size. It sizes the workspace.
 *   num_splits    as for sinkattn_prefill.
 *   workspace/workspace_bytes   device scratch, 256-byte aligned, at least
 *            sinkattn_prefill_paged_workspace_size() bytes for the same
 *            arguments (about batch * max_seqlen_k * hkv * 4 D bytes, plus
 *            the split partials); contents need not be initialised. The call
 *            first gathers every sequence's pages into contiguous rows there
 *            (K as bf16, V as fp16 for the P.V product, clamped to +-65504),
 *            then runs the prefill kernel on them.
 * A block-table entry outside [0, num_pages) or an Lk_b outside
 * [0, max_seqlen_k] is not read through: the key row is staged as zeros, or
 * the length clamped, and the device error word (sinkattn_get_device_error)
 * records code 2 or 3.
 */
size_t sinkattn_prefill_paged_workspace_size(int batch, int64_t total_q, int max_seqlen_q,
                                             int max_seqlen_k, int hq, int hkv, int head_dim,
                                             int window, int num_splits);

sinkattn_status_t sinkattn_prefill_paged(const void *q, const int32_t *cu_seqlens_q,
                                         const void *k_cache, const void *v_cache,
                                         const int32_t *block_table, const int32_t *seqlens_k,
                                         int num_pages, int max_pages_per_seq, int page_size,
                                         int batch, int64_t total_q, int max_seqlen_q,
                                         int max_seqlen_k, int hq, int hkv, int head_dim,
                                         const float *sinks, sinkattn_mask_t mask,
                                         int num_splits, void *out, float *lse, void *workspace,
                                         size_t workspace_bytes, void *stream);

/*
 * Prefill of packed queries against a paged fp8 KV cache (page "GPT-OSS on
 * day 0": the model is served with FP8; a chunked prefill then reads the
 * cache that decode reads). Same arguments, workspace
 * (sinkattn_prefill_paged_workspace_size), error reporting and results as
 * sinkattn_prefill_paged, except:
 *   k_cache, v_cache  fp8 e4m3 codes (the encoding of sinkattn_decode_fp8),
 *            one byte per element, [num_pages, hkv, page_size, D].
 *   k_scale, v_scale  float32 [hkv] or NULL (= 1): key j of KV head g stands
 *            for k_scale[g] * e4m3(k_cache[...]), likewise for v.
 * The gather stages the codes' exact values (K as bf16, V as fp16); k_scale
 * multiplies the softmax scale and v_scale the normalised output, so the
 * products are those of the bf16 call on the dequantised values up to the
 * rounding of scale * k_scale and of the final scaling.
 */
sinkattn_status_t sinkattn_prefill_paged_fp8(
    const void *q, const int32_t *cu_seqlens_q, const void *k_cache, const void *v_cache,
    const float *k_scale, const float *v_scale, const int32_t *block_table,
    const int32_t *seqlens_k, int num_pages, int max_pages_per_seq, int page_size, int batch,
    int64_t total_q, int max_seqlen_q, int max_seqlen_k, int hq, int hkv, int head_dim,
    const float *sinks, sinkattn_mask_t mask, int num_splits, void *out, float *lse,
    void *workspace, size_t workspace_bytes, void *stream);

/*
 * Decode: one query token per sequence over a KV cache, split along the KV
 * sequence (section "Kernels for GPT-OSS / Sink Attention": attention is
 * parallelised over heads and over the KV length; the sink enters one block
 * only). Block partials are merged by log-sum-exp inside the same launch: the
 * last block of each (sequence, KV head) to finish merges them.
 *
 *   q        bf16 [batch, hq, D]. The query sits at position Lk_b - 1.
 * Contiguous cache (block_table == NULL):
 *   k_cache, v_cache  bf16 [kv_rows, hkv, D]; sequence b owns rows
 *            kv_indptr[b]..kv_indptr[b+1]; kv_indptr int32 [batch+1], device,
 *            starting at 0; kv_rows = kv_indptr[batch] (host copy).
 *            seqlens_k must be NULL.
 * Paged cache (page "Fast embeddings on GPUs", section "ROSE": paged decode):
 *   k_cache, v_cache  bf16 [kv_rows, hkv, page_size, D]; kv_rows = number of
 *            pages. block_table int32 [batch, max_pages_per_seq], device:
 *            key j of sequence b is slot j % page_size of page
 *            block_table[b][j / page_size]. seqlens_k int32 [batch], device.
 *            kv_indptr must be NULL. Any page_size >= 1 works; 16 is the
 *            tested serving layout. The caller guarantees every entry the
 *            lengths reach is in [0, kv_rows) and seqlens_k[b] <=
 *            max_pages_per_seq * page_size: the decode kernel does not check
 *            them (checks measured 3-13% slower on the paged workloads).
 *   max_seqlen_k   host upper bound on Lk_b (sizes the split grid).
 *   num_splits     0 = automatic; n > 0 = split the longest sequence into
 *            about n blocks (shorter ones get proportionally fewer).
 *   hq / hkv: any group size. Up to 8 query heads share one read of each
 *            K/V row inside a block; larger groups are served in tiles of 8
 *            query heads, one block (or warp) per tile, whose reads of the same
 *            K/V rows are issued close together so that the repeats are
 *            served from L2.
 *   head_dim 64 or 128. q, out and every K/V row have head_dim elements.
 *   out      bf16 [batch, hq, D];  lse float32 [batch, hq] or NULL.
 *   workspace      device scratch of at least sinkattn_decode_workspace_size()
 *            bytes for the same (batch, max_seqlen_k, hq, hkv, head_dim,
 *            window, num_splits), 256-byte aligned; its contents need not be
 *            initialised and are overwritten. When the plan has a single block
 *            per sequence (short contexts or a short window) it is not touched
 *            and may be NULL.
 * mask.causal has no effect here (every cached key is at or before the query).
 */
size_t sinkattn_decode_workspace_size(int batch, int max_seqlen_k, int hq, int hkv, int head_dim,
                                      int window, int num_splits);

sinkattn_status_t sinkattn_decode(const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *kv_indptr, const int32_t *block_table,
                                  const int32_t *seqlens_k, int64_t kv_rows,
                                  int max_pages_per_seq, int page_size, int batch,
                                  int max_seqlen_k, int hq, int hkv, int head_dim,
                                  const float *sinks, sinkattn_mask_t mask, int num_splits,
                                  void *out, float *lse, void *workspace,
                                  size_t workspace_bytes, void *stream);

/*
 * Decode over an fp8 KV cache (page "GPT-OSS on day 0": the model is served
 * with FP8). Same arguments, layouts, plan, workspace
 * (sinkattn_decode_workspace_size) and results as sinkattn_decode, except:
 *   k_cache, v_cache  fp8 e4m3 (OCP "E4M3": 1 sign, 4 exponent bits with
 *            bias 7, 3 mantissa bits; 0x7F / 0xFF are NaN), one byte per
 *            element, with the same [rows, hkv, 64] or [pages, hkv, page, 64]
 *            layout; rows are 64 bytes.
 *   k_scale, v_scale  float32 [hkv] or NULL (= 1): key j of KV head g stands
 *            for k_scale[g] * e4m3(k_cache[...]), likewise for v.
 * The products run in fp16 (every e4m3 value is exact in fp16; q is rounded
 * to fp16, clamped to +-65504) with fp32 accumulation.
 */
sinkattn_status_t sinkattn_decode_fp8(const void *q, const void *k_cache, const void *v_cache,
                                      const float *k_scale, const float *v_scale,
                                      const int32_t *kv_indptr, const int32_t *block_table,
                                      const int32_t *seqlens_k, int64_t kv_rows,
                                      int max_pages_per_seq, int page_size, int batch,
                                      int max_seqlen_k, int hq, int hkv, int head_dim,
                                      const float *sinks, sinkattn_mask_t mask, int num_splits,
                                      void *out, float *lse, void *workspace,
                                      size_t workspace_bytes, void *stream);

/*
 * Allocation-free decode. The pages have no counterpart to this entry point;
 * it exists for callers that cannot give the library a scratch buffer:
 * code running under a memory planner that owns all device memory, plugin
 * hosts that forbid allocation while work is enqueued, and latency-critical
 * loops in which cudaMalloc/cudaFree could synchronise the device.
 *
 * Same arguments and results as sinkattn_decode, without the workspace: the
 * split-KV partials and counters live in a fixed device array of
 * SINKATTN_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that
 * loads the library holds until the process exits. The library still
 * allocates nothing at call time; the caller passes all inputs and outputs.
 *  - A plan whose scratch (sinkattn_decode_workspace_size for the same
 *    arguments) exceeds SINKATTN_NOALLOC_SCRATCH_BYTES is rejected with
 *    SINKATTN_ERR_WORKSPACE_TOO_SMALL before anything is enqueued (an
 *    explicit, smaller num_splits shrinks the scratch a batch needs).
 *  - The first call in each CUDA context (normally each device's primary
 *    context) looks up the array's device address with that context current;
 *    make that first call before any stream capture. A context created
 *    later (e.g. after cudaDeviceReset) gets its own lookup on its first call.
 *  - Failures of that lookup or of the launch return SINKATTN_ERR_CUDA and
 *    are reported by sinkattn_last_cuda_error, as for the other calls.
 *  - All calls on a device share the array and it keeps the last call's
 *    contents (counters are cleared on the stream by each call). Calls whose
 *    work can overlap on the GPU, e.g. on unordered streams, race on it.
 */
#define SINKATTN_NOALLOC_SCRATCH_BYTES (32u << 20)

sinkattn_status_t sinkattn_decode_noalloc(const void *q, const void *k_cache,
                                          const void *v_cache, const int32_t *kv_indptr,
                                          const int32_t *block_table, const int32_t *seqlens_k,
                                          int64_t kv_rows, int max_pages_per_seq, int page_size,
                                          int batch, int max_seqlen_k, int hq, int hkv,
                                          int head_dim, const float *sinks, sinkattn_mask_t mask,
                                          int num_splits, void *out, float *lse, void *stream);

/*
 * Merge of split-KV partials by log-sum-exp (section "Kernels for GPT-OSS /
 * Sink Attention": when the KV sequence is split into blocks, the sink belongs
 * to one block only; here it may enter as its own block, exactly once).
 *
 *   partial_o    float32 [num_splits, rows, hq, D]: each block's normalised output
 *   partial_lse  float32 [num_splits, rows, hq]: each block's natural-log lse;
 *                -inf marks an empty block (its partial_o is ignored).
 *   sinks        float32 [hq] or NULL; when given, the sink is one more block
 *                with lse = sinks[h] and a zero output.
 *   out          bf16 [rows, hq, D];   lse float32 [rows, hq] or NULL.
 * With M = max_k lse_k: out = sum_k e^{lse_k - M} o_k / sum_k e^{lse_k - M},
 * lse = M + ln sum_k e^{lse_k - M}. All blocks empty: out = 0, lse = -inf.
 */
sinkattn_status_t sinkattn_merge(const float *partial_o, const float *partial_lse,
                                 int num_splits, int64_t rows, int hq, int head_dim,
                                 const float *sinks, void *out, float *lse, void *stream);

/*
 * Backward of sinkattn_prefill (packed sequences, contiguous K/V). The pages
 * give the forward only; the gradients follow from its definition (section
 * "Kernels for GPT-OSS / Sink Attention": one sink logit per head in the
 * softmax denominator, no value row). With P_ij = e^{s_ij - lse_i},
 * P_sink,i = e^{sink_h - lse_i}, D_i = dO_i . O_i and
 * dS_ij = P_ij (dO_i . v_j - D_i):
 *   dq_i = scale sum_j dS_ij k_j,  dk_j = scale sum_i dS_ij q_i,
 *   dv_j = sum_i P_ij dO_i,         dsink_h = -sum_i P_sink,i D_i,
 * with dk, dv summed over the query heads sharing a KV head and dsink over
 * every row of head h.
 *
 *   q, k, v, cu_seqlens_*, total_*, max_seqlen_*, hq, hkv, head_dim, sinks,
 *            mask   exactly as passed to the forward call.
 *   out, lse       the forward's outputs for the same inputs (bf16
 *            [total_q, hq, 64]; float32 [total_q, hq], required).
 *   dout     bf16 [total_q, hq, 64]: gradient of the loss with respect to out.
 *   dq       bf16 [total_q, hq, 64];  dk, dv  bf16 [total_k, hkv, 64].
 *            Every element is written (rows that see no key get 0).
 *   dsinks   float32 [hq] or NULL; written when both sinks and dsinks are
 *            given.
 *   workspace/workspace_bytes   device scratch, 256-byte aligned, at least
 *            sinkattn_prefill_backward_workspace_size() bytes for the same
 *            sizes (fp16 copies of q, k, v and dout, two float32 values per
 *            (row, head), two tile lists); contents need not be initialised.
 * The products run on fp16 copies of the inputs (values of magnitude above
 * 65504 are clamped) with fp32 accumulation; P and dS enter the second
 * products as fp16. Every output element is written by one CTA, so repeated
 * calls give bitwise identical results.
 */
size_t sinkattn_prefill_backward_workspace_size(int batch, int64_t total_q, int64_t total_k,
                                                int hq, int hkv, int head_dim);

sinkattn_status_t sinkattn_prefill_backward(
    const void *q, const void *k, const void *v, const void *out, const void *dout,
    const float *lse, const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int batch,
    int64_t total_q, int64_t total_k, int max_seqlen_q, int max_seqlen_k, int hq, int hkv,
    int head_dim, const float *sinks, sinkattn_mask_t mask, void *dq, void *dk, void *dv,
    float *dsinks, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Device error word (prefill, paged prefill and backward kernels). Every
 * wait inside the kernels is bounded; a wait that
 * runs out records a nonzero code here and the kernel returns early instead of
 * hanging. This call synchronises `stream`, copies the word to *code and
 * resets it to 0. Codes: 0 none; 1 a pipeline barrier wait timed out;
 * 2 a paged-prefill block-table entry was outside [0, num_pages); 3 a length
 * above its host bound (a query length past max_seqlen_q in a prefill or
 * backward call, a key length past max_seqlen_k in a backward call, a
 * paged-prefill key length outside [0, max_seqlen_k]).
 */
sinkattn_status_t sinkattn_get_device_error(void *stream, int *code);

/*
 * Testing hook, not part of the computation: exercises the timeout path of
 * the bounded waits. With limit_ns > 0, every prefill, paged prefill and
 * backward call launched afterwards (in this process) makes one extra wait,
 * before the first scores of each CTA (the backward: of its dQ kernel), on a
 * barrier that nothing completes, bounded by limit_ns nanoseconds. Each CTA
 * then does what any timed-out wait makes it do: records code 1 in the
 * device error word, stops issuing work, waits (with the normal one-second
 * bound) for the copies and tensor-core products it already issued,
 * releases its tensor memory and exits. The outputs of such calls are
 * unspecified. limit_ns = 0 turns the hook off. The setting is read at
 * launch time (host side), so it is safe to change between launches.
 */
sinkattn_status_t sinkattn_debug_stall_waits(uint64_t limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* SINKATTN_H */
