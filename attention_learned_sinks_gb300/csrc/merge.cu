// Log-sum-exp merge of split-KV partials.
//
// Page "GPT-OSS on day 0", section "Kernels for GPT-OSS / Sink Attention":
// attention split along the KV sequence is recombined from per-block results,
// and the sink must be counted once. Here each block k brings a normalised
// output o_k and its natural-log lse_k; the optional sink is one more block
// with lse = sink_h and a zero output. One warp per (row, head); each lane
// owns two of the 64 output dims. HBM-bound: reads num_splits * 260 B and
// writes 132 B per (row, head).
#include <math.h>

#include "launch.h"
#include "ptx.cuh"

namespace sinkattn {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__global__ void __launch_bounds__(kWarpsPerBlock * 32) merge_kernel(
    const float *__restrict__ po, const float *__restrict__ pl, int nsplit, int64_t rows, int hq,
    const float *__restrict__ sinks, __nv_bfloat16 *__restrict__ out, float *__restrict__ lse) {
  const int64_t n = rows * hq;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  if (idx >= n) return;
  const int lane = threadIdx.x & 31;
  const int h = static_cast<int>(idx % hq);
  const float sink = sinks != nullptr ? sinks[h] : -INFINITY;

  float M = sink;
  for (int k = 0; k < nsplit; ++k) M = fmaxf(M, pl[k * n + idx]);
  float W = 0.f, a0 = 0.f, a1 = 0.f;
  if (M != -INFINITY) {
    W = sinks != nullptr ? fast_exp2((sink - M) * kLog2e) : 0.f;
    for (int k = 0; k < nsplit; ++k) {
      const float l = pl[k * n + idx];
      if (l == -INFINITY) continue;
      const float w = fast_exp2((l - M) * kLog2e);
      const float2 o = *reinterpret_cast<const float2 *>(po + (k * n + idx) * kHeadDim + 2 * lane);
      W += w;
      a0 += w * o.x;
      a1 += w * o.y;
    }
  }
  const float iw = W > 0.f ? 1.f / W : 0.f;
  reinterpret_cast<uint32_t *>(out + idx * kHeadDim)[lane] = pack_bf16x2(a0 * iw, a1 * iw);
  if (lse != nullptr && lane == 0) lse[idx] = W > 0.f ? M + fast_log2(W) * kLn2 : -INFINITY;
}

}  // namespace

cudaError_t launch_merge(const float *partial_o, const float *partial_lse, int num_splits,
                         int64_t rows, int hq, const float *sinks, void *out, float *lse,
                         cudaStream_t stream) {
  const int64_t n = rows * hq;
  if (n == 0) return cudaSuccess;
  const int64_t blocks = (n + kWarpsPerBlock - 1) / kWarpsPerBlock;
  merge_kernel<<<static_cast<unsigned>(blocks), kWarpsPerBlock * 32, 0, stream>>>(
      partial_o, partial_lse, num_splits, rows, hq, sinks, static_cast<__nv_bfloat16 *>(out), lse);
  return cudaGetLastError();
}

}  // namespace sinkattn
