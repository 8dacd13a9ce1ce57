// Log-sum-exp merge of split-KV partials.
//
// Page "GPT-OSS on day 0", section "Kernels for GPT-OSS / Sink Attention":
// attention split along the KV sequence is recombined from per-block results,
// and the sink must be counted once. Here each block k brings a normalised
// output o_k and its natural-log lse_k; the optional sink is one more block
// with lse = sink_h and a zero output. One warp per (row, head); each lane
// owns D/32 of the D output dims (D = 64 or 128). HBM-bound: reads
// num_splits * (4 D + 4) B and writes 2 D + 4 B per (row, head).
#include <math.h>

#include "launch.h"
#include "ptx.cuh"

namespace sinkattn {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
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
  constexpr int kPer = D / 32;  // dims per lane: 2 or 4
  float W = 0.f, acc[kPer] = {};
  if (M != -INFINITY) {
    W = sinks != nullptr ? fast_exp2((sink - M) * kLog2e) : 0.f;
    for (int k = 0; k < nsplit; ++k) {
      const float l = pl[k * n + idx];
      if (l == -INFINITY) continue;
      const float w = fast_exp2((l - M) * kLog2e);
      const float *o = po + (k * n + idx) * D + kPer * lane;
      float ov[kPer];
      if constexpr (kPer == 2) {
        const float2 t = *reinterpret_cast<const float2 *>(o);
        ov[0] = t.x, ov[1] = t.y;
      } else {
        const float4 t = *reinterpret_cast<const float4 *>(o);
        ov[0] = t.x, ov[1] = t.y, ov[2] = t.z, ov[3] = t.w;
      }
      W += w;
#pragma unroll
      for (int i = 0; i < kPer; ++i) acc[i] += w * ov[i];
    }
  }
  const float iw = W > 0.f ? 1.f / W : 0.f;
  uint32_t *dst = reinterpret_cast<uint32_t *>(out + idx * D) + (kPer / 2) * lane;
#pragma unroll
  for (int i = 0; i < kPer / 2; ++i) dst[i] = pack_bf16x2(acc[2 * i] * iw, acc[2 * i + 1] * iw);
  if (lse != nullptr && lane == 0) lse[idx] = W > 0.f ? M + fast_log2(W) * kLn2 : -INFINITY;
}

}  // namespace

cudaError_t launch_merge(const float *partial_o, const float *partial_lse, int num_splits,
                         int64_t rows, int hq, int head_dim, const float *sinks, void *out,
                         float *lse, cudaStream_t stream) {
  const int64_t n = rows * hq;
  if (n == 0) return cudaSuccess;
  const int64_t blocks = (n + kWarpsPerBlock - 1) / kWarpsPerBlock;
  auto *o = static_cast<__nv_bfloat16 *>(out);
  if (head_dim == 128)
    merge_kernel<128><<<static_cast<unsigned>(blocks), kWarpsPerBlock * 32, 0, stream>>>(
        partial_o, partial_lse, num_splits, rows, hq, sinks, o, lse);
  else
    merge_kernel<64><<<static_cast<unsigned>(blocks), kWarpsPerBlock * 32, 0, stream>>>(
        partial_o, partial_lse, num_splits, rows, hq, sinks, o, lse);
  return cudaGetLastError();
}

}  // namespace sinkattn
