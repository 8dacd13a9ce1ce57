// Prefill for sink attention over packed variable-length sequences, on the
// sm_103a tensor cores (tcgen05 + TMEM) with TMA-staged tiles.
//
// Page "GPT-OSS on day 0", section "Kernels for GPT-OSS / Sink Attention":
// an online softmax with running maximum m and denominator d, where m starts
// at the head's sink (d = 1) rather than at -inf. Page "Fast embeddings on
// GPUs", section "ROSE": attention on ragged inputs without padding
// (cu_seqlens). Page "CuTeDSL at Perplexity", section "Prefill and decode
// specialisation": prefill is compute-bound, so its kernel is built around
// the tensor cores.
//
// P V runs in fp16: P (in [0, 256], see the rescale rule below) keeps 11
// significant bits instead of bf16's 8, which keeps the output error near the
// bf16 rounding of the output itself. V is first converted to fp16 by a
// bandwidth-bound pre-pass into the caller's workspace (exact for every bf16
// value of magnitude up to 65504; larger ones clamp to +-65504). Q K^T stays
// in bf16.
//
// One CTA = 128 query rows of one (sequence, query head); 6 warps:
//   warps 0-3  softmax: thread r owns row r (TMEM lane r)
//   warp 4     TMA producer: Q once, then K_j / V_j into a 3-stage ring
//   warp 5     MMA issuer (one thread): S_j = Q K_j^T into TMEM (two S
//              buffers), O += P_j V_j with P_j read from TMEM
// TMEM (512 columns): S0 [0,128), S1 [128,256), O [256,320); P_j (bf16 pairs)
// overwrites the first 64 columns of its S buffer after S_j has been read.
// The running maximum is only moved (and O, d rescaled) when it grows by more
// than 8 in log2 units; the final division uses the same reference maximum,
// so the result is unchanged while most tiles skip the O round trip.
#include <math.h>

#include <mutex>

#include "launch.h"
#include "ptx.cuh"

namespace sinkattn {
namespace {

constexpr int kBM = 128;  // query rows per CTA
constexpr int kBN = 128;  // keys per KV tile
constexpr int kStages = 3;
constexpr int kTileBytes = kBM * kHeadDim * 2;  // 16 KB: 128 rows x 128 B
constexpr int kThreads = 192;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS0 = 0, kTmemO = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// shared memory map (offsets from a 1024-byte aligned base)
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileBytes;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kOffBar = kOffV + kStages * kTileBytes;
constexpr int kSmemBytes = kOffBar + 256 + 1024;  // + barriers + alignment slack

constexpr uint32_t kIdescQK = idesc_f32acc(kBM, kBN, /*bf16=*/true, false, false);
constexpr uint32_t kIdescPV = idesc_f32acc(kBM, kHeadDim, /*bf16=*/false, false, true);

__device__ int g_prefill_error;

struct Params {
  const int32_t *cu_q, *cu_k;
  int hq, group, causal, window, max_qtiles;
  const float *sinks;
  float scale_log2;
  __nv_bfloat16 *out;
  float *lse;
};

struct Barriers {
  uint64_t q_full;
  uint64_t k_full[kStages];
  uint64_t v_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Barriers) <= 256, "barrier block");

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (sbase - raw);
  Barriers *bars = reinterpret_cast<Barriers *>(smem + kOffBar);
  volatile int *abort = &bars->abort;

  const int h = blockIdx.x;
  const int b = blockIdx.y;
  const int qt = p.max_qtiles - 1 - static_cast<int>(blockIdx.z);  // longest work first
  const int q0 = p.cu_q[b], lq = p.cu_q[b + 1] - q0;
  const int k0 = p.cu_k[b], lk = p.cu_k[b + 1] - k0;
  if (qt * kBM >= lq) return;  // CTA-uniform
  const int rows = min(kBM, lq - qt * kBM);
  const int kvh = h / p.group;
  const int p_min = lk - lq + qt * kBM;  // position of this tile's first query
  const int p_max = p_min + rows - 1;
  int key_hi = lk;
  if (p.causal) key_hi = min(key_hi, p_max + 1);
  int key_lo = 0;
  if (p.window > 0) key_lo = max(0, p_min - p.window + 1);
  const int kt_lo = key_lo / kBN;
  const int n = key_hi > key_lo ? (key_hi + kBN - 1) / kBN - kt_lo : 0;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], kBM);
    }
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&bars->q_full, kTileBytes);
      tma_load_3d(sbase + kOffQ, &tm_q, &bars->q_full, 0, h, q0 + qt * kBM);
      int issued = 0;
      for (int j = 0; j < n; ++j) {
        const int st = j % kStages;
        if (j >= kStages &&
            !mbar_wait(&bars->kv_empty[st], ((j / kStages) - 1) & 1, abort, &g_prefill_error))
          break;
        const int row = k0 + (kt_lo + j) * kBN;
        mbar_arrive_expect_tx(&bars->k_full[st], kTileBytes);
        tma_load_3d(sbase + kOffK + st * kTileBytes, &tm_k, &bars->k_full[st], 0, kvh, row);
        mbar_arrive_expect_tx(&bars->v_full[st], kTileBytes);
        tma_load_3d(sbase + kOffV + st * kTileBytes, &tm_v, &bars->v_full[st], 0, kvh, row);
        issued = j + 1;
      }
      if (*abort) {
        // Copies already issued still land in this CTA's shared memory: wait
        // for them (bounded) before the CTA may exit.
        mbar_wait(&bars->q_full, 0, abort, &g_prefill_error, true);
        for (int j = max(0, issued - kStages); j < issued; ++j) {
          mbar_wait(&bars->k_full[j % kStages], (j / kStages) & 1, abort, &g_prefill_error, true);
          mbar_wait(&bars->v_full[j % kStages], (j / kStages) & 1, abort, &g_prefill_error, true);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && n > 0) {
      const uint64_t qdesc = sdesc_sw128(sbase + kOffQ);
      auto issue_pv = [&](int i) -> bool {
        if (!mbar_wait(&bars->p_full[i & 1], (i >> 1) & 1, abort, &g_prefill_error)) return false;
        if (!mbar_wait(&bars->v_full[i % kStages], (i / kStages) & 1, abort, &g_prefill_error))
          return false;
        tc_fence_after();
        const uint64_t vdesc = sdesc_sw128(sbase + kOffV + (i % kStages) * kTileBytes);
        const uint32_t pcol = tmem + kTmemS0 + (i & 1) * kBN;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          umma_ts(tmem + kTmemO, pcol + kk * 8, vdesc + ((kk * 16 * 128) >> 4), kIdescPV,
                  (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bars->kv_empty[i % kStages]);
        umma_commit(&bars->o_done);
        return true;
      };
      bool ok = mbar_wait(&bars->q_full, 0, abort, &g_prefill_error);
      for (int j = 0; ok && j < n; ++j) {
        const int st = j % kStages;
        if (!mbar_wait(&bars->k_full[st], (j / kStages) & 1, abort, &g_prefill_error)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t kdesc = sdesc_sw128(sbase + kOffK + st * kTileBytes);
        const uint32_t sbuf = tmem + kTmemS0 + (j & 1) * kBN;
#pragma unroll
        for (int ks = 0; ks < kHeadDim / 16; ++ks)
          umma_ss(sbuf, qdesc + ((ks * 32) >> 4), kdesc + ((ks * 32) >> 4), kIdescQK,
                  ks > 0 ? 1u : 0u);
        umma_commit(&bars->s_full[j & 1]);
        if (j > 0) ok = issue_pv(j - 1);
      }
      if (ok) issue_pv(n - 1);
      // every MMA issued by this thread has finished before TMEM is released
      umma_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, abort, &g_prefill_error, true);
    }
  } else {
    // -------------------------------------------------------------- softmax
    const int r = threadIdx.x;  // row within the tile == TMEM lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const bool has_sink = p.sinks != nullptr;
    float m_run = has_sink ? p.sinks[h] * kLog2e : -INFINITY;
    float d_run = has_sink ? 1.f : 0.f;
    const float c = p.scale_log2;
    const int pos = p_min + r;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int buf = j & 1;
      // waits are made warp-uniform: tcgen05.ld/st below are warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full[buf], (j >> 1) & 1, abort,
                                             &g_prefill_error))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[kBN];
#pragma unroll
      for (int q = 0; q < kBN / 32; ++q)
        tmem_ld32(lane_addr + kTmemS0 + buf * kBN + q * 32,
                  *reinterpret_cast<uint32_t(*)[32]>(&sr[q * 32]));
      tmem_wait_ld();
      float s[kBN];
#pragma unroll
      for (int i = 0; i < kBN; ++i) s[i] = __uint_as_float(sr[i]);

      const int key0 = (kt_lo + j) * kBN;
      const bool need_mask = (key0 + kBN > lk) || (p.causal && key0 + kBN - 1 > p_min) ||
                             (p.window > 0 && key0 <= p_max - p.window);
      if (need_mask) {
#pragma unroll
        for (int i = 0; i < kBN; ++i) {
          const int key = key0 + i;
          const bool vis = key < lk && (!p.causal || key <= pos) &&
                           (p.window == 0 || key > pos - p.window);
          if (!vis) s[i] = -INFINITY;
        }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < kBN; ++i) mx = fmaxf(mx, s[i]);
      const float m_tile = mx * c;
      const float m_new = fmaxf(m_run, m_tile);
      float alpha = 1.f;
      bool rescale = false;
      if (m_new > m_run + kRescaleThreshold) {
        alpha = fast_exp2(m_run - m_new);
        d_run *= alpha;
        m_run = m_new;
        rescale = true;
      }
      const float base = m_run == -INFINITY ? 0.f : m_run;
      float sum = 0.f;
      uint32_t pk[kBN / 2];
#pragma unroll
      for (int i = 0; i < kBN / 2; ++i) {
        const float p0 = fast_exp2(fmaf(s[2 * i], c, -base));
        const float p1 = fast_exp2(fmaf(s[2 * i + 1], c, -base));
        sum += p0 + p1;
        pk[i] = pack_f16x2(p0, p1);
      }
      d_run += sum;
#pragma unroll
      for (int q = 0; q < kBN / 64; ++q)
        tmem_st32(lane_addr + kTmemS0 + buf * kBN + q * 32,
                  *reinterpret_cast<uint32_t(*)[32]>(&pk[q * 32]));
      tmem_wait_st();
      if (j > 0) {
        // O holds P_0..P_{j-1} V; it must be complete before it is rescaled,
        // and waiting for every phase in order keeps the parity unambiguous.
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&bars->o_done, (j - 1) & 1, abort, &g_prefill_error))) {
          ok = false;
          break;
        }
        // one lane's rescale makes the whole warp run the (collective) O round
        // trip; lanes that did not move their maximum multiply by alpha = 1
        if (__any_sync(0xffffffffu, rescale)) {
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < kHeadDim / 32; ++q) {
            uint32_t ov[32];
            tmem_ld32(lane_addr + kTmemO + q * 32, ov);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(lane_addr + kTmemO + q * 32, ov);
          }
          tmem_wait_st();
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->p_full[buf]);
    }

    // ------------------------------------------------------------- epilogue
    float o[kHeadDim];
#pragma unroll
    for (int i = 0; i < kHeadDim; ++i) o[i] = 0.f;
    if (__all_sync(0xffffffffu,
                   ok && n > 0 && mbar_wait(&bars->o_done, (n - 1) & 1, abort, &g_prefill_error))) {
      tc_fence_after();
#pragma unroll
      for (int q = 0; q < kHeadDim / 32; ++q) {
        uint32_t ov[32];
        tmem_ld32(lane_addr + kTmemO + q * 32, ov);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) o[q * 32 + i] = __uint_as_float(ov[i]);
      }
    }
    if (r < rows) {
      const float inv = d_run > 0.f ? 1.f / d_run : 0.f;
      const size_t row_h = static_cast<size_t>(q0 + qt * kBM + r) * p.hq + h;
      uint4 *dst = reinterpret_cast<uint4 *>(p.out + row_h * kHeadDim);
#pragma unroll
      for (int i = 0; i < kHeadDim / 8; ++i) {
        uint4 v;
        v.x = pack_bf16x2(o[8 * i + 0] * inv, o[8 * i + 1] * inv);
        v.y = pack_bf16x2(o[8 * i + 2] * inv, o[8 * i + 3] * inv);
        v.z = pack_bf16x2(o[8 * i + 4] * inv, o[8 * i + 5] * inv);
        v.w = pack_bf16x2(o[8 * i + 6] * inv, o[8 * i + 7] * inv);
        dst[i] = v;
      }
      if (p.lse != nullptr)
        p.lse[row_h] = d_run > 0.f ? (m_run + fast_log2(d_run)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// bf16 V -> fp16 copy for the P V product (8 elements per thread per step).
__global__ void __launch_bounds__(256) convert_v_kernel(const uint4 *__restrict__ src,
                                                        uint4 *__restrict__ dst, int64_t n8) {
  const float lim = 65504.f;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 x = src[i];
    uint4 y;
    y.x = pack_f16x2(fminf(fmaxf(bf16_lo(x.x), -lim), lim), fminf(fmaxf(bf16_hi(x.x), -lim), lim));
    y.y = pack_f16x2(fminf(fmaxf(bf16_lo(x.y), -lim), lim), fminf(fmaxf(bf16_hi(x.y), -lim), lim));
    y.z = pack_f16x2(fminf(fmaxf(bf16_lo(x.z), -lim), lim), fminf(fmaxf(bf16_hi(x.z), -lim), lim));
    y.w = pack_f16x2(fminf(fmaxf(bf16_lo(x.w), -lim), lim), fminf(fmaxf(bf16_hi(x.w), -lim), lim));
    dst[i] = y;
  }
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// [rows, heads, 64] 16-bit tensor; a box is 128 rows of one head, 128-byte swizzle.
bool encode_rows_heads(EncodeTiledFn fn, CUtensorMap *map, const void *base, int64_t rows,
                       int heads, CUtensorMapDataType dtype) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(rows < 1 ? 1 : rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim * 2),
                                 static_cast<cuuint64_t>(heads) * kHeadDim * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kHeadDim), 1, static_cast<cuuint32_t>(kBM)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, dtype, 3, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t prefill_workspace_bytes(int64_t total_k, int hkv) {
  const size_t bytes = static_cast<size_t>(total_k) * hkv * kHeadDim * 2;
  return (bytes + 255) / 256 * 256;
}

cudaError_t launch_prefill(const PrefillLaunch &a, cudaStream_t stream, bool *encode_failed) {
  *encode_failed = false;
  const int max_qtiles = (a.max_seqlen_q + kBM - 1) / kBM;
  if (a.batch == 0 || a.total_q == 0 || max_qtiles == 0) return cudaSuccess;
  EncodeTiledFn fn = get_encode_fn();
  CUtensorMap tq, tk, tv;
  const CUtensorMapDataType bf16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  // With no keys at all nothing reads K or V; the maps then point at q.
  const void *kbase = a.total_k > 0 ? a.k : a.q;
  const void *vbase = a.total_k > 0 ? a.v_f16 : a.q;
  if (fn == nullptr || !encode_rows_heads(fn, &tq, a.q, a.total_q, a.hq, bf16) ||
      !encode_rows_heads(fn, &tk, kbase, a.total_k, a.hkv, bf16) ||
      !encode_rows_heads(fn, &tv, vbase, a.total_k, a.hkv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)) {
    *encode_failed = true;
    return cudaErrorInvalidValue;
  }
  const int64_t n8 = a.total_k * a.hkv * kHeadDim / 8;
  if (n8 > 0) {
    const int64_t blocks = (n8 + 255) / 256;
    convert_v_kernel<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(
        static_cast<const uint4 *>(a.v), static_cast<uint4 *>(a.v_f16), n8);
  }
  Params p;
  p.cu_q = a.cu_q;
  p.cu_k = a.cu_k;
  p.hq = a.hq;
  p.group = a.hq / a.hkv;
  p.causal = a.causal ? 1 : 0;
  p.window = a.window;
  p.max_qtiles = max_qtiles;
  p.sinks = a.sinks;
  p.scale_log2 = a.scale * kLog2e;
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.lse = a.lse;
  cudaError_t e =
      cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(a.hq, a.batch, max_qtiles);
  prefill_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

cudaError_t prefill_read_error(cudaStream_t stream, int *code) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(code, g_prefill_error, sizeof(int));
  const int zero = 0;
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof(int));
  return e;
}

}  // namespace sinkattn
