// Internal host interface between the C ABI (abi.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace sinkattn {

constexpr int kHeadDim = 64;

// Status code of the C ABI for a CUDA result (0 = ok); a failure is recorded
// as the calling thread's last CUDA error (sinkattn_last_cuda_error).
int cuda_status(cudaError_t e);

// ---- decode ----------------------------------------------------------------
// Split plan: the visible KV range of every (sequence, KV head) is cut into
// blocks of `chunk` tokens; max_splits bounds the block count of any sequence.
struct DecodePlan {
  int chunk;
  int max_splits;
};
// Query heads of a KV head are served in tiles of up to 8 (the MMA's N);
// groups above 8 take several tiles, each its own block (or warp).
inline int decode_head_tiles(int hq, int hkv) { return (hq / hkv + 7) / 8; }
DecodePlan plan_decode(int batch, int hq, int hkv, int max_seqlen_k, int window, int num_splits);
// Workspace layout for a plan: [partial_o | partial_lse | counters].
struct DecodeWorkspace {
  size_t off_lse, off_counters, bytes;
};
DecodeWorkspace decode_workspace_layout(int batch, int hq, int hkv, const DecodePlan &plan,
                                        int head_dim);
// head dims the decode kernels are built for
inline bool decode_head_dim_ok(int d) { return d == 64 || d == 128; }

struct DecodeLaunch {
  const void *q, *k, *v;  // k, v: bf16, or fp8 e4m3 bytes when fp8
  bool fp8 = false;
  const float *k_scale = nullptr, *v_scale = nullptr;  // fp8: per KV head (null = 1)
  int head_dim = kHeadDim;  // 64 or 128
  const int32_t *kv_indptr, *block_table, *seqlens_k;
  int max_pages, page_size;
  int batch, max_seqlen_k, hq, hkv, window;
  const float *sinks;
  float scale;
  void *out;
  float *lse;
  void *workspace;
  DecodePlan plan;
};
cudaError_t launch_decode(const DecodeLaunch &a, cudaStream_t stream);

// ---- merge -----------------------------------------------------------------
cudaError_t launch_merge(const float *partial_o, const float *partial_lse, int num_splits,
                         int64_t rows, int hq, int head_dim, const float *sinks, void *out,
                         float *lse, cudaStream_t stream);

// ---- tile lists ------------------------------------------------------------
// One block on `stream`: the non-empty (sequence b, 128-row tile t) pairs of
// the ragged layout cu[0..batch], packed b << 16 | t, tiles of higher index
// first (at most max_tiles per sequence); their count in *num_pairs; *counter
// zeroed. `pairs` holds up to cu[batch] / 128 + batch entries.
cudaError_t launch_tile_list(const int32_t *cu, int batch, int max_tiles, unsigned *pairs,
                             int *num_pairs, unsigned *counter, cudaStream_t stream);

// ---- prefill ---------------------------------------------------------------
struct PrefillLaunch {
  const void *q, *k, *v;
  const int32_t *cu_q, *cu_k;
  int batch;
  int64_t total_q, total_k;
  int max_seqlen_q, max_seqlen_k, hq, hkv;
  const float *sinks;
  int causal, window;
  float scale;
  void *out;
  float *lse;
  int num_splits;  // key-range splits per work item (>= 1), from prefill_plan_splits
  int head_dim = kHeadDim;  // 64 or 128
  // per-KV-head scales of fp8 K/V values (NULL: 1); set by the fp8 paged call
  const float *k_scale = nullptr, *v_scale = nullptr;
  // workspace (prefill_workspace_bytes): fp16 copy of v, tile counter, work
  // list, split partials
  void *v_f16;
};
// Key-range splits for a prefill call: requested > 0 is taken as is (capped at
// kMaxPrefillSplits); 0 picks a count from the host bounds so that calls with
// few (query tile, head) items over long contexts fill the GPU.
constexpr int kMaxPrefillSplits = 64;
int prefill_plan_splits(int requested, int batch, int64_t total_q, int max_seqlen_q,
                        int max_seqlen_k, int hq, int hkv, int window, int head_dim);
size_t prefill_workspace_bytes(int batch, int64_t total_q, int64_t total_k, int hq, int hkv,
                               int splits, int head_dim);
// head dims the prefill kernels are built for
inline bool prefill_head_dim_ok(int d) { return d == 64 || d == 128; }
// Returns cudaSuccess, or the failing CUDA error; *encode_failed is set when
// the tensor-map encoding (driver entry point) failed.
cudaError_t launch_prefill(const PrefillLaunch &a, cudaStream_t stream, bool *encode_failed);
// Prefill over a paged K/V cache: the referenced pages are gathered into
// contiguous staging (K bf16, V fp16) in the workspace, then the same kernel
// runs. base.k/v/cu_k/total_k/v_f16 are unused.
struct PrefillPagedLaunch {
  PrefillLaunch base;
  const void *k_cache, *v_cache;  // [num_pages, hkv, page_size, D] bf16, or e4m3 with fp8
  bool fp8 = false;
  const int32_t *block_table, *seqlens_k;
  int max_pages, page_size, num_pages;
  void *workspace;
};
size_t prefill_paged_workspace_bytes(int batch, int64_t total_q, int max_seqlen_k, int hq,
                                     int hkv, int splits, int head_dim);
cudaError_t launch_prefill_paged(const PrefillPagedLaunch &a, cudaStream_t stream,
                                 bool *encode_failed);
// ---- backward --------------------------------------------------------------
struct BackwardLaunch {
  const void *q, *k, *v, *out, *dout;  // bf16
  const float *lse;                    // [total_q, hq], natural log, sink included
  const int32_t *cu_q, *cu_k;
  int batch;
  int64_t total_q, total_k;
  int max_seqlen_q, max_seqlen_k, hq, hkv;
  const float *sinks;
  int causal, window;
  float scale;
  void *dq, *dk, *dv;  // bf16 [.., D]
  float *dsinks;       // [hq] or null
  void *workspace;     // backward_workspace_bytes
  int head_dim = kHeadDim;  // 64 or 128
};
size_t backward_workspace_bytes(int batch, int64_t total_q, int64_t total_k, int hq, int hkv,
                                int head_dim);
// head dims the backward kernels are built for
inline bool backward_head_dim_ok(int d) { return d == 64 || d == 128; }
cudaError_t launch_backward(const BackwardLaunch &a, cudaStream_t stream, bool *encode_failed);
cudaError_t backward_read_error(cudaStream_t stream, int *code);

// Reads and clears the prefill kernel's device error word (synchronises stream).
cudaError_t prefill_read_error(cudaStream_t stream, int *code);
// Testing hook: prefill / backward kernels launched from now on make one wait
// of at most ns nanoseconds on a barrier that nothing completes (0: off).
cudaError_t prefill_set_stall(uint64_t ns);
cudaError_t backward_set_stall(uint64_t ns);

}  // namespace sinkattn
