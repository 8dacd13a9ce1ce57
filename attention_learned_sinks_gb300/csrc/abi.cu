// C ABI of libsinkattn.so (declared in include/sinkattn.h): argument
// validation, split planning and dispatch to the kernels. No device memory is
// allocated and no stream is synchronised here (except by
// sinkattn_get_device_error, which exists to read a device word back).
#include <math.h>
#include <stdint.h>

#include "../../include/sinkattn.h"
#include "launch.h"

using namespace sinkattn;

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool mask_ok(const sinkattn_mask_t &m) {
  return m.window >= 0 && isfinite(m.scale) && m.scale > 0.f;
}

// The CUDA error behind the calling thread's last SINKATTN_ERR_CUDA.
thread_local cudaError_t t_last_cuda_error = cudaSuccess;

sinkattn_status_t from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return SINKATTN_OK;
  t_last_cuda_error = e;
  return SINKATTN_ERR_CUDA;
}

}  // namespace

namespace sinkattn {
int cuda_status(cudaError_t e) { return from_cuda(e); }
}  // namespace sinkattn

extern "C" {

const char *sinkattn_last_cuda_error(void) {
  return t_last_cuda_error == cudaSuccess ? "no CUDA error" : cudaGetErrorName(t_last_cuda_error);
}

const char *sinkattn_status_string(sinkattn_status_t s) {
  switch (s) {
    case SINKATTN_OK:
      return "ok";
    case SINKATTN_ERR_INVALID_ARGUMENT:
      return "invalid argument";
    case SINKATTN_ERR_UNSUPPORTED:
      return "unsupported configuration";
    case SINKATTN_ERR_WORKSPACE_TOO_SMALL:
      return "workspace too small";
    case SINKATTN_ERR_CUDA:
      return "CUDA error";
  }
  return "unknown status";
}

size_t sinkattn_prefill_workspace_size(int batch, int64_t total_q, int64_t total_k,
                                       int max_seqlen_q, int max_seqlen_k, int hq, int hkv,
                                       int head_dim, int window, int num_splits) {
  if (batch < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 ||
      hq <= 0 || hkv <= 0 || hq % hkv != 0 || !prefill_head_dim_ok(head_dim) || window < 0 ||
      num_splits < 0)
    return 0;
  const int splits = prefill_plan_splits(num_splits, batch, total_q, max_seqlen_q, max_seqlen_k,
                                         hq, hkv, window, head_dim);
  return prefill_workspace_bytes(batch, total_q, total_k, hq, hkv, splits, head_dim);
}

sinkattn_status_t sinkattn_prefill(const void *q, const void *k, const void *v,
                                   const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                   int batch, int64_t total_q, int64_t total_k, int max_seqlen_q,
                                   int max_seqlen_k, int hq, int hkv, int head_dim,
                                   const float *sinks, sinkattn_mask_t mask, int num_splits,
                                   void *out, float *lse, void *workspace, size_t workspace_bytes,
                                   void *stream) {
  if (batch < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || hq <= 0 ||
      hkv <= 0 || hq % hkv != 0 || num_splits < 0 || !mask_ok(mask))
    return SINKATTN_ERR_INVALID_ARGUMENT;
  if (!prefill_head_dim_ok(head_dim)) return SINKATTN_ERR_UNSUPPORTED;
  if (batch == 0 || total_q == 0 || max_seqlen_q == 0) return SINKATTN_OK;
  if (!q || !k || !v || !cu_seqlens_q || !cu_seqlens_k || !out)
    return SINKATTN_ERR_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4) || (sinks && !aligned(sinks, 4)) ||
      (lse && !aligned(lse, 4)))
    return SINKATTN_ERR_INVALID_ARGUMENT;
  if (batch > 65535 || hq > 65535 || total_q > INT32_MAX || total_k > INT32_MAX ||
      (max_seqlen_q + 127) / 128 > 65535)
    return SINKATTN_ERR_UNSUPPORTED;
  const int splits = prefill_plan_splits(num_splits, batch, total_q, max_seqlen_q, max_seqlen_k,
                                         hq, hkv, mask.window, head_dim);
  if (splits > 1 && static_cast<int64_t>(splits) * total_q * hq > INT32_MAX)
    return SINKATTN_ERR_UNSUPPORTED;
  const size_t need = prefill_workspace_bytes(batch, total_q, total_k, hq, hkv, splits, head_dim);
  if (workspace == nullptr || workspace_bytes < need) return SINKATTN_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(workspace, 256)) return SINKATTN_ERR_INVALID_ARGUMENT;
  PrefillLaunch a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.batch = batch;
  a.total_q = total_q;
  a.total_k = total_k;
  a.max_seqlen_q = max_seqlen_q;
  a.max_seqlen_k = max_seqlen_k;
  a.hq = hq;
  a.hkv = hkv;
  a.sinks = sinks;
  a.causal = mask.causal != 0;
  a.window = mask.window;
  a.scale = mask.scale;
  a.out = out;
  a.lse = lse;
  a.num_splits = splits;
  a.head_dim = head_dim;
  a.v_f16 = workspace;
  bool encode_failed = false;
  cudaError_t e = launch_prefill(a, static_cast<cudaStream_t>(stream), &encode_failed);
  if (encode_failed) return SINKATTN_ERR_CUDA;
  return from_cuda(e);
}

size_t sinkattn_prefill_paged_workspace_size(int batch, int64_t total_q, int max_seqlen_q,
                                             int max_seqlen_k, int hq, int hkv, int head_dim,
                                             int window, int num_splits) {
  if (batch < 0 || total_q < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || hq <= 0 || hkv <= 0 ||
      hq % hkv != 0 || !prefill_head_dim_ok(head_dim) || window < 0 || num_splits < 0)
    return 0;
  const int splits = prefill_plan_splits(num_splits, batch, total_q, max_seqlen_q, max_seqlen_k,
                                         hq, hkv, window, head_dim);
  return prefill_paged_workspace_bytes(batch, total_q, max_seqlen_k, hq, hkv, splits, head_dim);
}

}  // extern "C"

namespace {

sinkattn_status_t prefill_paged_impl(const void *q, const int32_t *cu_seqlens_q,
                                     const void *k_cache, const void *v_cache, bool fp8,
                                     const float *k_scale, const float *v_scale,
                                     const int32_t *block_table, const int32_t *seqlens_k,
                                     int num_pages, int max_pages_per_seq, int page_size,
                                     int batch, int64_t total_q, int max_seqlen_q,
                                     int max_seqlen_k, int hq, int hkv, int head_dim,
                                     const float *sinks, sinkattn_mask_t mask, int num_splits,
                                     void *out, float *lse, void *workspace,
                                     size_t workspace_bytes, void *stream) {
  if (batch < 0 || total_q < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || hq <= 0 || hkv <= 0 ||
      hq % hkv != 0 || num_pages < 0 || max_pages_per_seq < 0 || page_size <= 0 ||
      num_splits < 0 || !mask_ok(mask))
    return SINKATTN_ERR_INVALID_ARGUMENT;
  if (!prefill_head_dim_ok(head_dim)) return SINKATTN_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_seqlen_k) > static_cast<int64_t>(max_pages_per_seq) * page_size)
    return SINKATTN_ERR_INVALID_ARGUMENT;
  if (batch == 0 || total_q == 0 || max_seqlen_q == 0) return SINKATTN_OK;
  if (!q || !cu_seqlens_q || !seqlens_k || !out) return SINKATTN_ERR_INVALID_ARGUMENT;
  if (max_seqlen_k > 0 && (!k_cache || !v_cache || !block_table || num_pages == 0))
    return SINKATTN_ERR_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(cu_seqlens_q, 4) || !aligned(block_table, 4) || !aligned(seqlens_k, 4) ||
      (sinks && !aligned(sinks, 4)) || (lse && !aligned(lse, 4)) ||
      (k_scale && !aligned(k_scale, 4)) || (v_scale && !aligned(v_scale, 4)))
    return SINKATTN_ERR_INVALID_ARGUMENT;
  if (batch > 65535 || hq > 65535 || total_q > INT32_MAX || (max_seqlen_q + 127) / 128 > 65535 ||
      static_cast<int64_t>(batch) * max_seqlen_k + 128 > INT32_MAX)
    return SINKATTN_ERR_UNSUPPORTED;
  const int splits = prefill_plan_splits(num_splits, batch, total_q, max_seqlen_q, max_seqlen_k,
                                         hq, hkv, mask.window, head_dim);
  if (splits > 1 && static_cast<int64_t>(splits) * total_q * hq > INT32_MAX)
    return SINKATTN_ERR_UNSUPPORTED;
  const size_t need =
      prefill_paged_workspace_bytes(batch, total_q, max_seqlen_k, hq, hkv, splits, head_dim);
  if (workspace == nullptr || workspace_bytes < need) return SINKATTN_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(workspace, 256)) return SINKATTN_ERR_INVALID_ARGUMENT;
  PrefillPagedLaunch a;
  a.base.q = q;
  a.base.k = nullptr;
  a.base.v = nullptr;
  a.base.cu_q = cu_seqlens_q;
  a.base.cu_k = nullptr;
  a.base.batch = batch;
  a.base.total_q = total_q;
  a.base.total_k = 0;
  a.base.max_seqlen_q = max_seqlen_q;
  a.base.max_seqlen_k = max_seqlen_k;
  a.base.hq = hq;
  a.base.hkv = hkv;
  a.base.sinks = sinks;
  a.base.causal = mask.causal != 0;
  a.base.window = mask.window;
  a.base.scale = mask.scale;
  a.base.out = out;
  a.base.lse = lse;
  a.base.num_splits = splits;
  a.base.head_dim = head_dim;
  a.base.k_scale = k_scale;
  a.base.v_scale = v_scale;
  a.base.v_f16 = nullptr;
  a.fp8 = fp8;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = block_table;
  a.seqlens_k = seqlens_k;
  a.max_pages = max_pages_per_seq;
  a.page_size = page_size;
  a.num_pages = num_pages;
  a.workspace = workspace;
  bool encode_failed = false;
  cudaError_t e = launch_prefill_paged(a, static_cast<cudaStream_t>(stream), &encode_failed);
  if (encode_failed) return SINKATTN_ERR_CUDA;
  return from_cuda(e);
}

}  // namespace

extern "C" {

sinkattn_status_t sinkattn_prefill_paged(const void *q, const int32_t *cu_seqlens_q,
                                         const void *k_cache, const void *v_cache,
                                         const int32_t *block_table, const int32_t *seqlens_k,
                                         int num_pages, int max_pages_per_seq, int page_size,
                                         int batch, int64_t total_q, int max_seqlen_q,
                                         int max_seqlen_k, int hq, int hkv, int head_dim,
                                         const float *sinks, sinkattn_mask_t mask,
                                         int num_splits, void *out, float *lse, void *workspace,
                                         size_t workspace_bytes, void *stream) {
  return prefill_paged_impl(q, cu_seqlens_q, k_cache, v_cache, false, nullptr, nullptr,
                            block_table, seqlens_k, num_pages, max_pages_per_seq, page_size,
                            batch, total_q, max_seqlen_q, max_seqlen_k, hq, hkv, head_dim, sinks,
                            mask, num_splits, out, lse, workspace, workspace_bytes, stream);
}

sinkattn_status_t sinkattn_prefill_paged_fp8(
    const void *q, const int32_t *cu_seqlens_q, const void *k_cache, const void *v_cache,
    const float *k_scale, const float *v_scale, const int32_t *block_table,
    const int32_t *seqlens_k, int num_pages, int max_pages_per_seq, int page_size, int batch,
    int64_t total_q, int max_seqlen_q, int max_seqlen_k, int hq, int hkv, int head_dim,
    const float *sinks, sinkattn_mask_t mask, int num_splits, void *out, float *lse,
    void *workspace, size_t workspace_bytes, void *stream) {
  return prefill_paged_impl(q, cu_seqlens_q, k_cache, v_cache, true, k_scale, v_scale,
                            block_table, seqlens_k, num_pages, max_pages_per_seq, page_size,
                            batch, total_q, max_seqlen_q, max_seqlen_k, hq, hkv, head_dim, sinks,
                            mask, num_splits, out, lse, workspace, workspace_bytes, stream);
}

size_t sinkattn_decode_workspace_size(int batch, int max_seqlen_k, int hq, int hkv, int head_dim,
                                      int window, int num_splits) {
  if (batch <= 0 || hq <= 0 || hkv <= 0 || !decode_head_dim_ok(head_dim) || max_seqlen_k < 0 ||
      window < 0 || num_splits < 0)
    return 0;
  const DecodePlan plan = plan_decode(batch, hq, hkv, max_seqlen_k, window, num_splits);
  return decode_workspace_layout(batch, hq, hkv, plan, head_dim).bytes;
}

}  // extern "C"

namespace {

sinkattn_status_t decode_impl(const void *q, const void *k_cache, const void *v_cache, bool fp8,
                              const float *k_scale, const float *v_scale,
                              const int32_t *kv_indptr, const int32_t *block_table,
                              const int32_t *seqlens_k, int64_t kv_rows, int max_pages_per_seq,
                              int page_size, int batch, int max_seqlen_k, int hq, int hkv,
                              int head_dim, const float *sinks, sinkattn_mask_t mask,
                              int num_splits, void *out, float *lse, void *workspace,
                              size_t workspace_bytes, void *stream) {
  if (batch < 0 || max_seqlen_k < 0 || hq <= 0 || hkv <= 0 || hq % hkv != 0 || num_splits < 0 ||
      kv_rows < 0 || !mask_ok(mask))
    return SINKATTN_ERR_INVALID_ARGUMENT;
  if (!decode_head_dim_ok(head_dim)) return SINKATTN_ERR_UNSUPPORTED;
  const bool paged = block_table != nullptr;
  if (paged == (kv_indptr != nullptr)) return SINKATTN_ERR_INVALID_ARGUMENT;
  if (paged && (seqlens_k == nullptr || page_size <= 0 || max_pages_per_seq <= 0))
    return SINKATTN_ERR_INVALID_ARGUMENT;
  if (!paged && seqlens_k != nullptr) return SINKATTN_ERR_INVALID_ARGUMENT;
  if (batch == 0) return SINKATTN_OK;
  if (!q || !k_cache || !v_cache || !out) return SINKATTN_ERR_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      (kv_indptr && !aligned(kv_indptr, 4)) || (block_table && !aligned(block_table, 4)) ||
      (seqlens_k && !aligned(seqlens_k, 4)) || (sinks && !aligned(sinks, 4)) ||
      (lse && !aligned(lse, 4)) || (k_scale && !aligned(k_scale, 4)) ||
      (v_scale && !aligned(v_scale, 4)))
    return SINKATTN_ERR_INVALID_ARGUMENT;
  if (batch > 65535 || static_cast<int64_t>(hkv) * decode_head_tiles(hq, hkv) > 65535)
    return SINKATTN_ERR_UNSUPPORTED;
  const DecodePlan plan = plan_decode(batch, hq, hkv, max_seqlen_k, mask.window, num_splits);
  if (plan.max_splits > 1) {
    const size_t need = decode_workspace_layout(batch, hq, hkv, plan, head_dim).bytes;
    if (workspace == nullptr || workspace_bytes < need) return SINKATTN_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(workspace, 256)) return SINKATTN_ERR_INVALID_ARGUMENT;
  }
  DecodeLaunch a;
  a.q = q;
  a.k = k_cache;
  a.v = v_cache;
  a.kv_indptr = kv_indptr;
  a.block_table = block_table;
  a.seqlens_k = seqlens_k;
  a.max_pages = max_pages_per_seq;
  a.page_size = page_size;
  a.batch = batch;
  a.max_seqlen_k = max_seqlen_k;
  a.hq = hq;
  a.hkv = hkv;
  a.window = mask.window;
  a.sinks = sinks;
  a.scale = mask.scale;
  a.out = out;
  a.lse = lse;
  a.workspace = workspace;
  a.plan = plan;
  a.fp8 = fp8;
  a.head_dim = head_dim;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  return from_cuda(launch_decode(a, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

sinkattn_status_t sinkattn_decode(const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *kv_indptr, const int32_t *block_table,
                                  const int32_t *seqlens_k, int64_t kv_rows, int max_pages_per_seq,
                                  int page_size, int batch, int max_seqlen_k, int hq, int hkv,
                                  int head_dim, const float *sinks, sinkattn_mask_t mask,
                                  int num_splits, void *out, float *lse, void *workspace,
                                  size_t workspace_bytes, void *stream) {
  return decode_impl(q, k_cache, v_cache, false, nullptr, nullptr, kv_indptr, block_table,
                     seqlens_k, kv_rows, max_pages_per_seq, page_size, batch, max_seqlen_k, hq,
                     hkv, head_dim, sinks, mask, num_splits, out, lse, workspace,
                     workspace_bytes, stream);
}

sinkattn_status_t sinkattn_decode_fp8(const void *q, const void *k_cache, const void *v_cache,
                                      const float *k_scale, const float *v_scale,
                                      const int32_t *kv_indptr, const int32_t *block_table,
                                      const int32_t *seqlens_k, int64_t kv_rows,
                                      int max_pages_per_seq, int page_size, int batch,
                                      int max_seqlen_k, int hq, int hkv, int head_dim,
                                      const float *sinks, sinkattn_mask_t mask, int num_splits,
                                      void *out, float *lse, void *workspace,
                                      size_t workspace_bytes, void *stream) {
  return decode_impl(q, k_cache, v_cache, true, k_scale, v_scale, kv_indptr, block_table,
                     seqlens_k, kv_rows, max_pages_per_seq, page_size, batch, max_seqlen_k, hq,
                     hkv, head_dim, sinks, mask, num_splits, out, lse, workspace,
                     workspace_bytes, stream);
}

sinkattn_status_t sinkattn_merge(const float *partial_o, const float *partial_lse, int num_splits,
                                 int64_t rows, int hq, int head_dim, const float *sinks, void *out,
                                 float *lse, void *stream) {
  if (num_splits < 0 || rows < 0 || hq <= 0) return SINKATTN_ERR_INVALID_ARGUMENT;
  if (!prefill_head_dim_ok(head_dim)) return SINKATTN_ERR_UNSUPPORTED;
  if (rows == 0) return SINKATTN_OK;
  if (!out || (num_splits > 0 && (!partial_o || !partial_lse)))
    return SINKATTN_ERR_INVALID_ARGUMENT;
  if ((partial_o && !aligned(partial_o, 16)) || (partial_lse && !aligned(partial_lse, 4)) ||
      !aligned(out, 16) || (sinks && !aligned(sinks, 4)) || (lse && !aligned(lse, 4)))
    return SINKATTN_ERR_INVALID_ARGUMENT;
  if ((rows * hq + 7) / 8 > INT32_MAX) return SINKATTN_ERR_UNSUPPORTED;
  return from_cuda(launch_merge(partial_o, partial_lse, num_splits, rows, hq, head_dim, sinks, out,
                                lse, static_cast<cudaStream_t>(stream)));
}

size_t sinkattn_prefill_backward_workspace_size(int batch, int64_t total_q, int64_t total_k,
                                                int hq, int hkv, int head_dim) {
  if (batch < 0 || total_q < 0 || total_k < 0 || hq <= 0 || hkv <= 0 || hq % hkv != 0 ||
      !backward_head_dim_ok(head_dim))
    return 0;
  return backward_workspace_bytes(batch, total_q, total_k, hq, hkv, head_dim);
}

sinkattn_status_t sinkattn_prefill_backward(
    const void *q, const void *k, const void *v, const void *out, const void *dout,
    const float *lse, const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int batch,
    int64_t total_q, int64_t total_k, int max_seqlen_q, int max_seqlen_k, int hq, int hkv,
    int head_dim, const float *sinks, sinkattn_mask_t mask, void *dq, void *dk, void *dv,
    float *dsinks, void *workspace, size_t workspace_bytes, void *stream) {
  if (batch < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || hq <= 0 ||
      hkv <= 0 || hq % hkv != 0 || !mask_ok(mask))
    return SINKATTN_ERR_INVALID_ARGUMENT;
  if (!backward_head_dim_ok(head_dim)) return SINKATTN_ERR_UNSUPPORTED;
  if (batch == 0 || (total_q == 0 && total_k == 0)) return SINKATTN_OK;
  if (!q || !k || !v || !out || !dout || !lse || !cu_seqlens_q || !cu_seqlens_k || !dq || !dk ||
      !dv)
    return SINKATTN_ERR_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(lse, 4) || !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4) ||
      (sinks && !aligned(sinks, 4)) || (dsinks && !aligned(dsinks, 4)))
    return SINKATTN_ERR_INVALID_ARGUMENT;
  if (batch > 65535 || total_q > INT32_MAX || total_k > INT32_MAX ||
      (max_seqlen_q + 127) / 128 > 65535 || (max_seqlen_k + 127) / 128 > 65535 ||
      (total_q / 128 + batch) * hq * (head_dim / 64) > INT32_MAX ||
      (total_k / 128 + batch) * hkv * (head_dim / 64) > INT32_MAX)
    return SINKATTN_ERR_UNSUPPORTED;
  const size_t need = backward_workspace_bytes(batch, total_q, total_k, hq, hkv, head_dim);
  if (workspace == nullptr || workspace_bytes < need) return SINKATTN_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(workspace, 256)) return SINKATTN_ERR_INVALID_ARGUMENT;
  BackwardLaunch a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.dout = dout;
  a.lse = lse;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.batch = batch;
  a.total_q = total_q;
  a.total_k = total_k;
  a.max_seqlen_q = max_seqlen_q;
  a.max_seqlen_k = max_seqlen_k;
  a.hq = hq;
  a.hkv = hkv;
  a.sinks = sinks;
  a.causal = mask.causal != 0;
  a.window = mask.window;
  a.scale = mask.scale;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dsinks = dsinks;
  a.workspace = workspace;
  a.head_dim = head_dim;
  bool encode_failed = false;
  cudaError_t e = launch_backward(a, static_cast<cudaStream_t>(stream), &encode_failed);
  if (encode_failed) return SINKATTN_ERR_CUDA;
  return from_cuda(e);
}

sinkattn_status_t sinkattn_debug_stall_waits(uint64_t limit_ns) {
  cudaError_t e = prefill_set_stall(limit_ns);
  if (e == cudaSuccess) e = backward_set_stall(limit_ns);
  return from_cuda(e);
}

sinkattn_status_t sinkattn_get_device_error(void *stream, int *code) {
  if (code == nullptr) return SINKATTN_ERR_INVALID_ARGUMENT;
  *code = 0;
  int other = 0;
  cudaError_t e = prefill_read_error(static_cast<cudaStream_t>(stream), code);
  if (e == cudaSuccess) e = backward_read_error(static_cast<cudaStream_t>(stream), &other);
  if (*code == 0) *code = other;
  return from_cuda(e);
}

}  // extern "C"
