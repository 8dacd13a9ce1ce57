// Backward pass of sink attention over packed variable-length sequences.
//
// The pages give the forward only (page "GPT-OSS on day 0", sections
// "Attention: GQA with Attention Sinks" and "Kernels for GPT-OSS / Sink
// Attention": one learned logit per head inside the softmax denominator, no
// value row). Its gradients, for row i of head h with P_j = e^{s_j - lse_i}
// (lse includes the sink) and P_c = e^{c_h - lse_i}:
//
//   D_i  = dO_i . O_i            dP_ij = dO_i . v_j
//   dS_ij = P_ij (dP_ij - D_i)
//   dq_i = scale sum_j dS_ij k_j     dk_j = scale sum_i dS_ij q_i
//   dv_j = sum_i P_ij dO_i           dc_h = -sum_i P_c,i D_i
//
// dk and dv of a KV head sum over its query heads. Launches, in order:
//  1. bwd_prep_q_kernel: fp16 copies of q and dO, D from the bf16 forward
//     output and lse in log2 units (head-major, so one tile's rows of one
//     head are contiguous);
//  2. bwd_prep_kv_kernel: fp16 copies of k and v;
//  3. two tile lists (query tiles, key tiles);
//  4. bwd_dq_kernel: persistent; per (query tile, head) item and key tile,
//     S = Q K^T and dP = dO V^T on tcgen05 into TMEM, P and dS in registers,
//     dQ += dS K (dS as the TMEM A operand) and Y += P K; it also forms the
//     exact D = sum_j P_j dP_j and corrects dQ with it;
//  5. bwd_dsink_kernel: dc_h, one block per head, fixed summation order;
//  6. bwd_dkdv_kernel: persistent; per (key tile, KV head) item and (query
//     head, query tile) step, S^T = K Q^T and dP^T = V dO^T, P^T and dS^T in
//     registers, dV += P^T dO and dK += dS^T Q with P^T / dS^T as TMEM A
//     operands.
// head_dim 128 (D = 128): the same kernels with items that also carry a
// 64-dimension half h of the output gradient: S and dP run over all 128
// dimensions (eight k-steps over two 64-column swizzle blocks), dQ, Y, dK and
// dV accumulate dimensions 64h..64h+63 (the K, Q and dO tiles' block h as the
// B operand), so the TMEM plan of D = 64 is kept; the two halves of one tile
// recompute S and dP. The exact D of a row is then written to its own array
// (both halves read the forward's D first). Shared memory: one Q/dO buffer
// and a two-stage K/V ring (dQ), one K/V buffer and a two-stage Q/dO ring
// (dK/dV).
// Every gradient element is written by exactly one CTA (no atomics), so the
// results are deterministic. All MMA operands are fp16 (bf16 inputs convert
// exactly except below 2^-14, and P, dS in fp16 keep 11 significant bits);
// accumulation is fp32. Every mbarrier wait is bounded.
#include <math.h>

#include <atomic>

#include "launch.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace sinkattn {
namespace {

constexpr int kBM = 128;                        // query rows per tile
constexpr int kBN = 128;                        // keys per tile
constexpr int kBlockBytes = 128 * 64 * 2;       // 16 KB: 128 rows x 64 dims, one swizzle block
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

// ts: A from TMEM, B MN-major in shared memory (dQ += dS K, ...), 64 output
// dimensions per product. fp16 inputs.
constexpr uint32_t kIdescTS = idesc_f32acc(128, 64, /*bf16=*/false, false, true);
constexpr uint64_t kBlockDesc = kBlockBytes >> 4;      // one 64-dim block in descriptor units
constexpr uint64_t kRows16Desc = (16 * 128) >> 4;      // 16 rows of 128 B

// one 128-row tile of one head at head dimension D (D / 64 swizzle blocks)
template <int D>
struct TileShape {
  static constexpr int kHalves = D / 64;  // 64-dim halves of an output gradient
  static constexpr int kBytes = 128 * D * 2;
  static constexpr uint64_t kDesc = kBytes >> 4;
};
// k-step ks of a D-dim K-major product: swizzle block ks / 4, 32-byte step ks % 4
__device__ __forceinline__ uint64_t kstep_off(int ks) {
  return (ks >> 2) * kBlockDesc + 2 * (ks & 3);
}

__device__ int g_backward_error;
// testing hook (sinkattn_debug_stall_waits): stall_ns of later launches
std::atomic<uint64_t> g_bwd_stall_ns{0};

struct BwdParams {
  const int32_t *cu_q, *cu_k;
  int batch, hq, hkv, group, causal, window;
  int total_q;
  float scale, scale_log2;
  // Per (head, row) vectors, stored negated so that the dK/dV kernel's copies
  // of a tile's 128 entries are the softmax-side operands as they stand:
  const float *nl2t;  // [hq][total_q]: -lse * log2(e) (-inf: row with no key and no sink)
  float *ndt;         // [hq][total_q]: -D from the forward output
  float *nde;         // [hq][total_q]: -(exact D) (dQ kernel; the same array as ndt at D = 64)
  const unsigned *q_pairs, *k_pairs;
  const int *num_q_pairs, *num_k_pairs;
  unsigned *q_counter, *k_counter;  // work counters of the persistent kernels (zeroed by the lists)
  __nv_bfloat16 *dq, *dk, *dv;
  // Testing hook (0: off): the dQ kernel's softmax-side warps wait at most
  // stall_ns on a barrier that nothing completes before their first scores,
  // so that every CTA of that kernel takes its timeout path.
  uint64_t stall_ns;
};

// ----------------------------------------------------------------- prep ---
// Thread = 8 consecutive elements of one (row, head), D / 8 threads a row.
// Every iteration of the block loop is uniform across the block, so the
// D / 8-lane shuffles always see full warps.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_q_kernel(
    const uint4 *__restrict__ q, const uint4 *__restrict__ dout, const uint4 *__restrict__ out,
    const float *__restrict__ lse, int64_t total_q, int hq, uint4 *__restrict__ q16,
    uint4 *__restrict__ do16, float *__restrict__ nl2t, float *__restrict__ ndt) {
  constexpr int kPer = D / 8;  // threads per (row, head)
  const int64_t n = total_q * hq * kPer;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x; base < n;
       base += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t i = base + threadIdx.x;
    float part = 0.f;
    if (i < n) {
      q16[i] = bf16x8_to_f16x8(q[i]);
      const uint4 g = dout[i], o = out[i];
      do16[i] = bf16x8_to_f16x8(g);
      part = bf16_lo(g.x) * bf16_lo(o.x) + bf16_hi(g.x) * bf16_hi(o.x) +
             bf16_lo(g.y) * bf16_lo(o.y) + bf16_hi(g.y) * bf16_hi(o.y) +
             bf16_lo(g.z) * bf16_lo(o.z) + bf16_hi(g.z) * bf16_hi(o.z) +
             bf16_lo(g.w) * bf16_lo(o.w) + bf16_hi(g.w) * bf16_hi(o.w);
    }
#pragma unroll
    for (int o = kPer / 2; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (i < n && (i % kPer) == 0) {
      const int64_t rh = i / kPer;
      const int64_t row = rh / hq;
      const int h = static_cast<int>(rh % hq);
      const float l = lse[rh];
      nl2t[h * total_q + row] = l == -INFINITY ? -INFINITY : -(l * kLog2e);
      ndt[h * total_q + row] = -part;
    }
  }
}

__global__ void __launch_bounds__(256) bwd_prep_kv_kernel(const uint4 *__restrict__ k,
                                                          const uint4 *__restrict__ v,
                                                          uint4 *__restrict__ k16,
                                                          uint4 *__restrict__ v16, int64_t n8) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    k16[i] = bf16x8_to_f16x8(k[i]);
    v16[i] = bf16x8_to_f16x8(v[i]);
  }
}

// dc_h = -sum_i e^{c_h - lse_i} D_i over every row of head h; double
// accumulation in a fixed order (per-thread strides, then a fixed tree).
__global__ void __launch_bounds__(256) bwd_dsink_kernel(const float *__restrict__ sinks,
                                                        const float *__restrict__ nl2t,
                                                        const float *__restrict__ ndt,
                                                        int64_t total_q,
                                                        float *__restrict__ dsinks) {
  // the dK/dV kernel does not read dsinks: it may start at once
  asm volatile("griddepcontrol.launch_dependents;");
  __shared__ double part[256];
  const int h = blockIdx.x;
  const float c2 = sinks[h] * kLog2e;
  double acc = 0.0;
  for (int64_t r = threadIdx.x; r < total_q; r += blockDim.x) {
    const float nl2 = nl2t[h * total_q + r];  // -lse log2(e); the second factor is -D
    if (nl2 != -INFINITY) acc += static_cast<double>(exp2f(c2 + nl2)) * ndt[h * total_q + r];
  }
  part[threadIdx.x] = acc;
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if (threadIdx.x < s) part[threadIdx.x] += part[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) dsinks[h] = static_cast<float>(part[0]);
}

// 32 columns of scores s (raw q.k) and dP -> P = 2^(s c - l2) (0 outside the
// visible range) and dS = P (dP - D), both packed as fp16 pairs. The per-row
// variant (dQ) takes l2 and D as scalars and also sums P dP into acc; the
// per-column one (dK/dV) takes them per column.
__device__ __forceinline__ void p_ds_row(float (&s)[32], const float (&dp)[32], float c, float l2,
                                         float d, uint32_t (&p16)[16], uint32_t (&ds16)[16],
                                         float2 &acc) {
  const float2 c2 = make_float2(c, c), nl = make_float2(-l2, -l2), nd = make_float2(-d, -d);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float2 a = __ffma2_rn(make_float2(s[2 * i], s[2 * i + 1]), c2, nl);
    const float2 p = make_float2(fast_exp2(a.x), fast_exp2(a.y));
    const float2 x = make_float2(dp[2 * i], dp[2 * i + 1]);
    const float2 ds = __fmul2_rn(p, __fadd2_rn(x, nd));
    acc = __ffma2_rn(p, x, acc);
    p16[i] = pack_f16x2(p.x, p.y);
    ds16[i] = pack_f16x2(ds.x, ds.y);
  }
}

// nl2 / nd: the columns' -l2 and -D (16-byte aligned shared memory)
__device__ __forceinline__ void p_ds_col(float (&s)[32], const float (&dp)[32], float c,
                                         const float *nl2, const float *nd, uint32_t (&p16)[16],
                                         uint32_t (&ds16)[16]) {
  const float2 c2 = make_float2(c, c);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 l = *reinterpret_cast<const float4 *>(nl2 + 4 * i);
    const float4 dd = *reinterpret_cast<const float4 *>(nd + 4 * i);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = 4 * i + 2 * h;
      const float2 a = __ffma2_rn(make_float2(s[j], s[j + 1]), c2,
                                  h == 0 ? make_float2(l.x, l.y) : make_float2(l.z, l.w));
      const float2 p = make_float2(fast_exp2(a.x), fast_exp2(a.y));
      const float2 g = __fadd2_rn(make_float2(dp[j], dp[j + 1]),
                                  h == 0 ? make_float2(dd.x, dd.y) : make_float2(dd.z, dd.w));
      const float2 ds = __fmul2_rn(p, g);
      p16[j / 2] = pack_f16x2(p.x, p.y);
      ds16[j / 2] = pack_f16x2(ds.x, ds.y);
    }
  }
}

// ---------------------------------------------------------------- dQ -------
// Persistent: one CTA per SM takes (query tile, head) items from the query
// tile list (longest first) through a global counter. Per 128-key tile,
// S = Q K^T and dP = dO V^T are single N = 128 products; softmax-side
// warpgroup w (warps 4w..4w+3, one query row per thread) turns keys
// 64w..64w+63 into P and dS. The warpgroups release S / dP as soon as they
// have loaded them, so the next tile's S and dP are computed while they
// work, and dQ / Y of a tile run while the next one is being softmaxed.
// Warp 8: TMA (Q and dO double-buffered per item, K/V in a 4-stage ring at
// head_dim 64, 2 stages at 128);
// warp 9: issues S and dP and owns TMEM; warp 10: issues dQ and Y.
//
// TMEM columns: S [0, 128), dP [128, 256), dS fp16 [256, 320), P fp16
// [320, 384) (warpgroup w's keys in the half at 32w), dQ [384, 448),
// Y [448, 512). S / dP of tile g are written only after both warpgroups have
// loaded those of tile g - 1, and dS / P of tile g only after the dQ / Y
// MMAs of tile g - 1 have completed; dQ and Y of an item start only after the
// previous item's epilogue has read them.
//
// D from the bf16 forward output (D_a) carries the output's rounding, and
// dP - D cancels when one key dominates a row. This kernel therefore also
// sums the exact D_e = sum_j P_j dP_j (fp32) and Y = sum_j P_j k_j (one more
// product), and corrects: dq = scale (sum_j P_j (dP_j - D_a) k_j
// - (D_e - D_a) Y). The correction is small, so its own fp16 rounding does
// not matter. D_e replaces D_a in the workspace for the dK/dV kernel and the
// sink gradient, which run after this one.
constexpr int kHalf = 64;  // keys (dK/dV: queries) of a tile per softmax warpgroup
// ss: both operands K-major in shared memory, 128 x 128 scores (S = Q K^T, ...)
constexpr uint32_t kIdescSS128 = idesc_f32acc(128, kBN, /*bf16=*/false, false, false);
constexpr int kDqThreads = 352;
constexpr int kDqStages = 4;  // K/V ring at D = 64 (the array size of the barriers)

// Shared memory of the dQ kernel: Q/dO buffers (two at D = 64, one at 128),
// the K/V ring (four stages at 64, two at 128), then the control block.
template <int D>
struct DqCfg {
  static constexpr int kTile = TileShape<D>::kBytes;
  static constexpr int kQdBufs = D == 64 ? 2 : 1;
  static constexpr int kStages = D == 64 ? 4 : 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kQdBufs * 2 * kTile;
  static constexpr int kOffV = kOffK + kStages * kTile;
  static constexpr int kOffBar = kOffV + kStages * kTile;
  static constexpr int kOffVec = kOffBar + 4096;  // per tile slot: -l2, -D of its 128 rows
  static constexpr int kSmem = kOffVec + 2048 + 1024;
};

struct DqTile {
  int valid, b, qt, h, g, q0, lq, k0, lk, rows, p_min, kt_lo, n, half;
};

struct DqBars {
  uint64_t tile_full[2], tile_empty[2];
  uint64_t qd_full[2], qd_empty[2];
  uint64_t kv_full[kDqStages], kv_empty[kDqStages];
  uint64_t s_full;    // S, dP of the current key tile are in TMEM
  uint64_t s_read;    // both warpgroups have loaded them (the buffers may be rewritten)
  uint64_t ds_full;   // both warpgroups have written dS, P of the tile
  uint64_t pds_free;  // dQ / Y of the tile have read dS, P
  uint64_t dq_done, dq_free, drain[2];
  uint64_t dsum_full[2];  // both warpgroups' partial sums of an item are in dsum
  uint64_t never;         // testing hook: a barrier nothing completes
  uint32_t tmem_base;
  int abort;
  DqTile tiles[2];
  float dsum[2][2][128];  // [item parity][warpgroup][row]: partial exact D
};

static_assert(sizeof(DqBars) <= 4096, "dQ control block");
static_assert(DqCfg<64>::kSmem <= 227 * 1024, "dQ shared memory at head_dim 64");
static_assert(DqCfg<128>::kSmem <= 227 * 1024, "dQ shared memory at head_dim 128");

// work index w -> item: 64-dim half w % halves of the output, then
// (sequence, query tile) list entry (w / halves) / hq and head (w / halves) % hq
__device__ __forceinline__ void dq_decode(const BwdParams &p, int halves, int w, DqTile &t) {
  t.half = w % halves;
  w /= halves;
  const unsigned e = p.q_pairs[w / p.hq];
  t.valid = 1;
  t.h = w % p.hq;
  t.g = t.h / p.group;
  t.b = static_cast<int>(e >> 16);
  t.qt = static_cast<int>(e & 0xffffu);
  t.q0 = p.cu_q[t.b];
  t.lq = p.cu_q[t.b + 1] - t.q0;
  t.k0 = p.cu_k[t.b];
  t.lk = p.cu_k[t.b + 1] - t.k0;
  t.rows = min(kBM, t.lq - t.qt * kBM);
  t.p_min = t.lk - t.lq + t.qt * kBM;
  const int p_max = t.p_min + t.rows - 1;
  int key_hi = t.lk, key_lo = 0;
  if (p.causal) key_hi = min(key_hi, p_max + 1);
  if (p.window > 0) key_lo = max(0, t.p_min - p.window + 1);
  t.kt_lo = key_lo / kBN;
  t.n = key_hi > key_lo ? (key_hi + kBN - 1) / kBN - t.kt_lo : 0;
}

// kV8 (both gradient kernels): dq, dk and dv start on 32-byte boundaries, and
// each thread's row segment is stored with 32-byte stores (whole sectors, half
// the store instructions); otherwise with 16-byte ones.
template <int D, bool kV8>
__global__ void __launch_bounds__(kDqThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const BwdParams p) {
  using C = DqCfg<D>;
  constexpr int kTileBytes = C::kTile;
  constexpr uint64_t kTileDesc = TileShape<D>::kDesc;
  constexpr int kHalves = TileShape<D>::kHalves;
  constexpr int kQdBufs = C::kQdBufs, kStages = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  DqBars *bars = reinterpret_cast<DqBars *>(smem_raw + (sbase - raw) + C::kOffBar);
  volatile int *abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int *err = &g_backward_error;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->tile_full[i], 1);
      mbar_init(&bars->tile_empty[i], 256 + 2);
      mbar_init(&bars->qd_full[i], 1);
      mbar_init(&bars->qd_empty[i], 1);
      mbar_init(&bars->drain[i], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_read, 256);
    mbar_init(&bars->ds_full, 256);
    mbar_init(&bars->pds_free, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 2);  // both MMA warps
    }
    mbar_init(&bars->dq_done, 1);
    mbar_init(&bars->dq_free, 256);
    mbar_init(&bars->dsum_full[0], 256);
    mbar_init(&bars->dsum_full[1], 256);
    mbar_init(&bars->never, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    const int num_work = *p.num_q_pairs * p.hq * kHalves;
    // one tile = D / 64 boxes of 64 dims into consecutive swizzle blocks
    auto load_tile = [&](uint32_t dst, const CUtensorMap *map, uint64_t *bar, int head, int row) {
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk)
        tma_load_3d_elect(dst + blk * kBlockBytes, map, bar, blk * 64, head, row);
    };
    int J = 0, nq = 0;
    bool ok = true;
    for (int nt = 0; ok; ++nt) {
      const int slot = nt & 1;
      if (nt >= 2 && !mbar_wait_warp(&bars->tile_empty[slot], ((nt >> 1) - 1) & 1, abort, err))
        break;
      if (lane == 0) {
        DqTile t;
        t.valid = 0;
        const int w = static_cast<int>(atomicAdd(p.q_counter, 1u));
        if (w < num_work) dq_decode(p, kHalves, w, t);
        bars->tiles[slot] = t;
      }
      __syncwarp();
      const DqTile t = bars->tiles[slot];
      // head_dim 64: the item's rows' -l2 / -D for the softmax warps, copied
      // ahead and tracked by the descriptor's barrier (rows past the tile read
      // as 0), so that an item's first step does not wait for two global
      // loads (3.45 -> 3.39 ms on the varlen backward; at head_dim 128 the
      // softmax warps load them themselves, 10.64 vs 10.70 ms)
      if (D == 64 && t.valid && t.n > 0) {
        const uint32_t vs = sbase + C::kOffVec + slot * 1024;
        const size_t at = static_cast<size_t>(t.h) * p.total_q + t.q0 + t.qt * kBM;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = lane + 32 * i;
          const bool in = row < t.rows;
          cp_async_4(vs + 4 * row, p.nl2t + at + (in ? row : 0), in ? 4u : 0u);
          cp_async_4(vs + 512 + 4 * row, p.ndt + at + (in ? row : 0), in ? 4u : 0u);
        }
        cp_async_mbar_arrive(&bars->tile_full[slot]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->tile_full[slot]);
      if (!t.valid) break;
      if (t.n == 0) continue;  // nothing to load (and no MMAs) for this item
      const int qb = nq % kQdBufs;
      if (nq >= kQdBufs &&
          !mbar_wait_warp(&bars->qd_empty[qb], ((nq / kQdBufs) - 1) & 1, abort, err))
        break;
      mbar_arrive_expect_tx_elect(&bars->qd_full[qb], 2 * kTileBytes);
      load_tile(sbase + C::kOffQ + qb * 2 * kTileBytes, &tm_q, &bars->qd_full[qb], t.h,
                t.q0 + t.qt * kBM);
      load_tile(sbase + C::kOffQ + (qb * 2 + 1) * kTileBytes, &tm_do, &bars->qd_full[qb], t.h,
                t.q0 + t.qt * kBM);
      ++nq;
      for (int j = 0; j < t.n; ++j, ++J) {
        const int st = J % kStages;
        if (J >= kStages &&
            !mbar_wait_warp(&bars->kv_empty[st], ((J / kStages) - 1) & 1, abort, err)) {
          ok = false;
          break;
        }
        const int row = t.k0 + (t.kt_lo + j) * kBN;
        mbar_arrive_expect_tx_elect(&bars->kv_full[st], 2 * kTileBytes);
        load_tile(sbase + C::kOffK + st * kTileBytes, &tm_k, &bars->kv_full[st], t.g, row);
        load_tile(sbase + C::kOffV + st * kTileBytes, &tm_v, &bars->kv_full[st], t.g, row);
      }
    }
    if (*abort) {  // copies already issued still land here: wait for them (bounded)
      for (int i = max(0, nq - kQdBufs); i < nq; ++i)
        mbar_wait_warp(&bars->qd_full[i % kQdBufs], (i / kQdBufs) & 1, abort, err, true);
      for (int i = max(0, J - kStages); i < J; ++i)
        mbar_wait_warp(&bars->kv_full[i % kStages], (i / kStages) & 1, abort, err, true);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // the vector copies have landed
  } else if (warp == 9 || warp == 10) {
    // ------------------------------------------------------------------ MMA
    // Two issuing warps, so that neither kind of product waits behind the
    // other in one instruction stream: warp 9 issues S = Q K^T and
    // dP = dO V^T of a key tile (N = 128) as soon as both softmax warpgroups
    // have loaded the previous tile's; warp 10 issues dQ += dS K and
    // Y += P K once they have written dS and P.
    const uint64_t kdesc0 = sdesc_sw128(sbase + C::kOffK);
    int J = 0, nq = 0;  // K/V tiles (= global tile index), items with keys
    int dq_items = 0;   // items whose dQ/Y the epilogue has to release
    bool ok = true;
    const bool is_s = warp == 9;
    const uint64_t qdesc0 = sdesc_sw128(sbase + C::kOffQ);
    const uint64_t vdesc0 = sdesc_sw128(sbase + C::kOffV);
    const uint32_t t_dq = tmem + 384, t_y = tmem + 448;
    for (int nt = 0; ok; ++nt) {
      const int slot = nt & 1;
      if (!mbar_wait_warp(&bars->tile_full[slot], (nt >> 1) & 1, abort, err)) break;
      const DqTile t = bars->tiles[slot];
      if (!t.valid) break;
      if (t.n > 0) {
        const int qb = nq % kQdBufs;
        if (is_s) {
          ok = mbar_wait_warp(&bars->qd_full[qb], (nq / kQdBufs) & 1, abort, err);
          for (int j = 0; ok && j < t.n; ++j) {
            const int g = J + j, st = g % kStages;
            // the softmax warps have loaded S / dP of tile g - 1
            if (!mbar_wait_warp(&bars->kv_full[st], (g / kStages) & 1, abort, err) ||
                (g >= 1 && !mbar_wait_warp(&bars->s_read, (g - 1) & 1, abort, err))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t qd = qdesc0 + qb * 2 * kTileDesc, dod = qd + kTileDesc;
            const uint64_t kd = kdesc0 + st * kTileDesc;
            const uint64_t vd = vdesc0 + st * kTileDesc;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              umma_ss_elect(tmem, qd + kstep_off(ks), kd + kstep_off(ks), kIdescSS128,
                            ks > 0 ? 1u : 0u);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              umma_ss_elect(tmem + 128, dod + kstep_off(ks), vd + kstep_off(ks), kIdescSS128,
                            ks > 0 ? 1u : 0u);
            umma_commit_elect(&bars->s_full);
            umma_commit_elect(&bars->kv_empty[st]);  // this warp is done with K/V
          }
          if (ok) umma_commit_elect(&bars->qd_empty[qb]);
        } else {
          // dQ/Y of the previous item must have been read by its epilogue
          if (dq_items > 0) ok = mbar_wait_warp(&bars->dq_free, (dq_items - 1) & 1, abort, err);
          for (int j = 0; ok && j < t.n; ++j) {
            const int g = J + j, st = g % kStages;
            if (!mbar_wait_warp(&bars->ds_full, g & 1, abort, err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // dims 64 half .. of K: the tile's swizzle block `half`
            const uint64_t kd = kdesc0 + st * kTileDesc + t.half * kBlockDesc;
            // dS / P of keys 0..127 are 64 consecutive fp16-pair columns
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              umma_ts_elect(t_dq, tmem + 256 + kk * 8, kd + kk * kRows16Desc, kIdescTS,
                            (j > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              umma_ts_elect(t_y, tmem + 320 + kk * 8, kd + kk * kRows16Desc, kIdescTS,
                            (j > 0 || kk > 0) ? 1u : 0u);
            umma_commit_elect(&bars->pds_free);  // dS / P may be overwritten
            umma_commit_elect(&bars->kv_empty[st]);
          }
          if (ok) umma_commit_elect(&bars->dq_done);
          ++dq_items;
        }
        if (!ok) break;
        ++nq;
        J += t.n;
      }
      if (lane == 0) mbar_arrive(&bars->tile_empty[slot]);
    }
    // every MMA issued by this warp has finished before TMEM is released
    umma_commit_elect(&bars->drain[warp - 9]);
    mbar_wait_warp(&bars->drain[warp - 9], 0, abort, err, true);
  } else {
    // ---------------------------------------- P, dS (one query row / thread)
    const int wg = warp >> 2;             // warpgroup: keys 64 wg .. 64 wg + 63 of each tile
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_off + 64 * wg, t_dp = t_s + 128;
    const uint32_t t_ds = tmem + lane_off + 256 + 32 * wg, t_p = t_ds + 64;
    const uint32_t t_dq = tmem + lane_off + 384 + 32 * wg, t_y = t_dq + 64;
    int G = 0, dq_items = 0;
    // testing hook: a wait that runs out while the first copies and products
    // are in flight
    bool ok = p.stall_ns == 0 || mbar_wait_warp(&bars->never, 0, abort, err, false, p.stall_ns);
    // An item's epilogue (exact D, dQ from TMEM, store) runs after the next
    // item's first dS / P have been handed to the tensor core: the item's last
    // dQ / Y products then complete while this warpgroup already computes, and
    // the next item's scores are not held up behind the stores. The pending
    // item's row, D and flags are kept here; its partial exact-D sums wait in
    // the dsum buffer of its parity.
    bool pend_on = false, pend_row = false, pend_de = false;
    __nv_bfloat16 *pend_dq = nullptr;
    size_t pend_lidx = 0;
    float pend_d = 0.f;
    auto finish = [&]() {
      const int par = dq_items & 1;
      if (!mbar_wait_warp(&bars->dsum_full[par], (dq_items >> 1) & 1, abort, err)) {
        ok = false;
        return;
      }
      const float *xs = bars->dsum[par][0];
      const float d_e = xs[r] + xs[128 + r];
      const float corr = d_e - pend_d;
      if (!mbar_wait_warp(&bars->dq_done, par, abort, err)) {
        ok = false;
        return;
      }
      ++dq_items;
      tc_fence_after();
      float a[32], y[32];
      tmem_ld32f(t_dq, a);
      tmem_ld32f(t_y, y);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars->dq_free);  // the next item's dQ / Y may start
      if (pend_row) {
        if constexpr (kV8) {
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              w[e] = pack_bf16x2(p.scale * fmaf(-corr, y[16 * i + 2 * e], a[16 * i + 2 * e]),
                                 p.scale * fmaf(-corr, y[16 * i + 2 * e + 1], a[16 * i + 2 * e + 1]));
            st_global_v8(pend_dq + 16 * i, w);
          }
        } else {
          uint4 *d4 = reinterpret_cast<uint4 *>(pend_dq);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = p.scale * fmaf(-corr, y[8 * i + e], a[8 * i + e]);
            d4[i] = make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]),
                               pack_bf16x2(o[4], o[5]), pack_bf16x2(o[6], o[7]));
          }
        }
        if (pend_de) p.nde[pend_lidx] = -d_e;
      }
      pend_on = false;
    };
    for (int nt = 0; ok; ++nt) {
      const int slot = nt & 1;
      if (!mbar_wait_warp(&bars->tile_full[slot], (nt >> 1) & 1, abort, err)) break;
      const DqTile t = bars->tiles[slot];
      if (!t.valid) break;
      const size_t qrow = static_cast<size_t>(t.q0 + t.qt * kBM + r);
      const size_t lidx = static_cast<size_t>(t.h) * p.total_q + qrow;
      __nv_bfloat16 *dq_row = p.dq + (qrow * p.hq + t.h) * D + 64 * t.half + 32 * wg;
      if (t.n == 0) {  // no row of this tile sees a key: dq = 0, D = 0
        if (r < t.rows) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            reinterpret_cast<uint4 *>(dq_row)[i] = make_uint4(0u, 0u, 0u, 0u);
          if (wg == 0 && t.half == 0) p.nde[lidx] = 0.f;
        }
        mbar_arrive(&bars->tile_empty[slot]);
        continue;
      }
      const float *vec =
          reinterpret_cast<const float *>(smem_raw + (sbase - raw) + C::kOffVec + slot * 1024);
      const float l2 = r >= t.rows ? INFINITY : D == 64 ? -vec[r] : -p.nl2t[lidx];
      const float d = r >= t.rows ? 0.f : D == 64 ? -vec[128 + r] : -p.ndt[lidx];
      const int pos = t.p_min + r;
      int hi = t.lk, lo = 0;
      if (p.causal) hi = min(hi, pos + 1);
      if (p.window > 0) lo = max(lo, pos - p.window + 1);
      if (r >= t.rows) hi = lo = 0;
      float2 dsum = make_float2(0.f, 0.f);
      // per key tile: this warpgroup's 64 keys (64 wg .. 64 wg + 63) in two
      // 32-column chunks; S / dP are released once both chunks are loaded
      for (int j = 0; j < t.n; ++j) {
        const int g = G + j;
        if (!mbar_wait_warp(&bars->s_full, g & 1, abort, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int key0 = (t.kt_lo + j) * kBN + wg * kHalf;
        const int c_lo = min(max(lo - key0, 0), kHalf);
        const int len = max(min(hi - key0, kHalf) - c_lo, 0);
        // 32-column chunks that some row of the warp does not see whole only
        // (warp-uniform, so the loads stay collective)
        const int end = c_lo + len;
        const bool mask_a = !__all_sync(0xffffffffu, c_lo <= 0 && end >= 32);
        const bool mask_b = !__all_sync(0xffffffffu, c_lo <= 32 && end >= 64);
        uint32_t p16a[16], ds16a[16];
        {
          float sv[32], dp[32];
          tmem_ld32f(t_s, sv);
          tmem_ld32f(t_dp, dp);
          tmem_wait_ld();
          if (mask_a) mask32(sv, 0, c_lo, len);
          p_ds_row(sv, dp, p.scale_log2, l2, d, p16a, ds16a, dsum);
        }
        float sv[32], dp[32];
        tmem_ld32f(t_s + 32, sv);
        tmem_ld32f(t_dp + 32, dp);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars->s_read);  // S / dP of the next tile may be computed
        if (mask_b) mask32(sv, 32, c_lo, len);
        uint32_t p16b[16], ds16b[16];
        p_ds_row(sv, dp, p.scale_log2, l2, d, p16b, ds16b, dsum);
        // dQ / Y of tile g - 1 have finished reading dS / P
        if (g >= 1) {
          if (!mbar_wait_warp(&bars->pds_free, (g - 1) & 1, abort, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        tmem_st16(t_ds, ds16a);
        tmem_st16(t_p, p16a);
        tmem_st16(t_ds + 16, ds16b);
        tmem_st16(t_p + 16, p16b);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->ds_full);
        if (j == 0 && pend_on) {
          finish();
          if (!ok) break;
        }
      }
      if (!ok) break;
      G += t.n;
      // exact D = both warpgroups' partial sums of P dP (exchanged through
      // shared memory; a bounded mbarrier wait, so an aborting CTA cannot
      // leave the other warpgroup waiting)
      (&bars->dsum[dq_items & 1][0][0])[wg * 128 + r] = dsum.x + dsum.y;
      mbar_arrive(&bars->dsum_full[dq_items & 1]);
      pend_on = true;
      pend_row = r < t.rows;
      pend_de = wg == 0 && t.half == 0;
      pend_dq = dq_row;
      pend_lidx = lidx;
      pend_d = d;
      mbar_arrive(&bars->tile_empty[slot]);
    }
    if (ok && pend_on) finish();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------- dK / dV -----
// Persistent: one CTA per SM takes (key tile, KV head) items from the key
// tile list (walked backwards: under a causal mask the low key tiles are seen
// by the most queries, so this is longest first within each KV head). An
// item's steps run over (query head of the group, query tile that sees the
// key tile). Per step, S^T = K Q^T and dP^T = V dO^T are single N = 128
// products; softmax-side warpgroup w (one key per thread) turns queries
// 64w..64w+63 into P^T and dS^T and releases S^T / dP^T once it has loaded
// them, so the next step's products are computed while it works. Warp 8: TMA
// (K/V double-buffered per item; Q, dO and the step's -lse / -D vectors in a
// 4-stage ring at head_dim 64, 2 stages at 128); warp 9: issues S^T and dP^T and owns TMEM; warp 10: issues
// dV and dK.
//
// TMEM columns: S^T [0, 128), dP^T [128, 256), P^T fp16 [256, 320), dS^T
// fp16 [320, 384) (warpgroup w's queries in the half at 32w), dV [384, 448),
// dK [448, 512).
constexpr int kKvThreads = 352;
constexpr int kKvQStages = 4;  // Q/dO ring at D = 64 (the array size of the barriers)

// Shared memory of the dK/dV kernel: K/V item buffers (two at D = 64, one at
// 128), the Q/dO ring (four stages at 64, two at 128) with each stage's
// -lse / -D vectors, then the control block.
template <int D>
struct KvCfg {
  static constexpr int kTile = TileShape<D>::kBytes;
  static constexpr int kKvBufs = D == 64 ? 2 : 1;
  static constexpr int kStages = D == 64 ? 4 : 2;
  static constexpr int kOffK = 0;
  static constexpr int kOffQ = kKvBufs * 2 * kTile;
  static constexpr int kOffVec = kOffQ + kStages * 2 * kTile;
  static constexpr int kOffBar = kOffVec + kStages * 1024;
  static constexpr int kSmem = kOffBar + 1024 + 1024;
};
static_assert(KvCfg<64>::kSmem <= 227 * 1024, "dK/dV shared memory at head_dim 64");
static_assert(KvCfg<128>::kSmem <= 227 * 1024, "dK/dV shared memory at head_dim 128");

struct KvTile {
  int valid, b, kt, g, q0, lq, k0, lk, krows, qt_lo, nqt, steps, half;
};

struct KvBars {
  uint64_t tile_full[2], tile_empty[2];
  uint64_t kv_full[2], kv_empty[2];
  uint64_t qd_full[kKvQStages], qd_empty[kKvQStages];
  uint64_t st_full;   // S^T, dP^T of the current step are in TMEM
  uint64_t s_read;    // both warpgroups have loaded them
  uint64_t ew_done;   // both warpgroups have written P^T, dS^T of the step
  uint64_t pds_free;  // dV / dK of the step have read P^T, dS^T
  uint64_t dkv_done, dkv_free, drain[2];
  uint32_t tmem_base;
  int abort;
  KvTile tiles[2];
};

static_assert(sizeof(KvBars) <= 1024, "dK/dV control block");

// Items are KV-head major: the CTAs in flight at one time work on key tiles
// of one KV head, so the Q / dO tiles of that head's query heads that they
// all stream stay in L2 between them (KV-head minor, every concurrent CTA
// streamed a different head: 10 GB from DRAM per call instead of 0.8 GB).
// With 64-dim halves, work index w -> half w % halves, then (w / halves) as
// above.
__device__ __forceinline__ void kv_decode(const BwdParams &p, int npairs, int halves, int w,
                                          KvTile &t) {
  t.half = w % halves;
  w /= halves;
  const unsigned e = p.k_pairs[npairs - 1 - w % npairs];
  t.valid = 1;
  t.g = w / npairs;
  t.b = static_cast<int>(e >> 16);
  t.kt = static_cast<int>(e & 0xffffu);
  t.q0 = p.cu_q[t.b];
  t.lq = p.cu_q[t.b + 1] - t.q0;
  t.k0 = p.cu_k[t.b];
  t.lk = p.cu_k[t.b + 1] - t.k0;
  t.krows = min(kBN, t.lk - t.kt * kBN);
  const int base = t.lk - t.lq;  // position of query 0
  const int jmin = t.kt * kBN, jmax = jmin + t.krows - 1;
  int iq_lo = 0, iq_hi = t.lq;   // queries that see at least one key of the tile
  if (p.causal) iq_lo = max(0, jmin - base);
  if (p.window > 0) iq_hi = min(iq_hi, jmax + p.window - base);
  t.qt_lo = iq_lo / kBM;
  t.nqt = iq_hi > iq_lo ? (iq_hi + kBM - 1) / kBM - t.qt_lo : 0;
  t.steps = t.nqt * p.group;
}

template <int D, bool kV8>
__global__ void __launch_bounds__(kKvThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const BwdParams p) {
  using C = KvCfg<D>;
  constexpr int kTileBytes = C::kTile;
  constexpr uint64_t kTileDesc = TileShape<D>::kDesc;
  constexpr int kHalves = TileShape<D>::kHalves;
  constexpr int kKvBufs = C::kKvBufs, kQStages = C::kStages;
  constexpr int kKvOffK = C::kOffK, kKvOffQ = C::kOffQ, kKvOffVec = C::kOffVec;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (sbase - raw);
  KvBars *bars = reinterpret_cast<KvBars *>(smem + C::kOffBar);
  volatile int *abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int *err = &g_backward_error;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->tile_full[i], 1);
      mbar_init(&bars->tile_empty[i], 256 + 2);
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
      mbar_init(&bars->drain[i], 1);
    }
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&bars->qd_full[s], 1);
      mbar_init(&bars->qd_empty[s], 2);  // both MMA warps
    }
    mbar_init(&bars->st_full, 1);
    mbar_init(&bars->s_read, 256);
    mbar_init(&bars->ew_done, 256);
    mbar_init(&bars->pds_free, 1);
    mbar_init(&bars->dkv_done, 1);
    mbar_init(&bars->dkv_free, 256);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    const int npairs = *p.num_k_pairs;
    const int num_work = npairs * p.hkv * kHalves;
    auto load_tile = [&](uint32_t dst, const CUtensorMap *map, uint64_t *bar, int head, int row) {
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk)
        tma_load_3d_elect(dst + blk * kBlockBytes, map, bar, blk * 64, head, row);
    };
    int ni = 0, S = 0;  // items with work, steps so far
    bool ok = true;
    for (int nt = 0; ok; ++nt) {
      const int slot = nt & 1;
      if (nt >= 2 && !mbar_wait_warp(&bars->tile_empty[slot], ((nt >> 1) - 1) & 1, abort, err))
        break;
      if (lane == 0) {
        KvTile t;
        t.valid = 0;
        const int w = static_cast<int>(atomicAdd(p.k_counter, 1u));
        if (w < num_work) kv_decode(p, npairs, kHalves, w, t);
        bars->tiles[slot] = t;
        mbar_arrive(&bars->tile_full[slot]);
      }
      __syncwarp();
      const KvTile t = bars->tiles[slot];
      if (!t.valid) break;
      if (t.steps == 0) continue;
      const int kb = ni % kKvBufs;
      if (ni >= kKvBufs &&
          !mbar_wait_warp(&bars->kv_empty[kb], ((ni / kKvBufs) - 1) & 1, abort, err))
        break;
      mbar_arrive_expect_tx_elect(&bars->kv_full[kb], 2 * kTileBytes);
      load_tile(sbase + kKvOffK + kb * 2 * kTileBytes, &tm_k, &bars->kv_full[kb], t.g,
                t.k0 + t.kt * kBN);
      load_tile(sbase + kKvOffK + (kb * 2 + 1) * kTileBytes, &tm_v, &bars->kv_full[kb], t.g,
                t.k0 + t.kt * kBN);
      ++ni;
      for (int s = 0; s < t.steps; ++s, ++S) {
        const int st = S % kQStages;
        const int h = t.g * p.group + s / t.nqt, qt = t.qt_lo + s % t.nqt;
        if (S >= kQStages &&
            !mbar_wait_warp(&bars->qd_empty[st], ((S / kQStages) - 1) & 1, abort, err)) {
          ok = false;
          break;
        }
        // -l2 / -D of the tile's 128 query rows, copied asynchronously and
        // tracked by the stage's barrier (the pending count each lane adds is
        // released when its copies land). Rows past the sequence read as 0:
        // their columns are masked, so P and dS are 0 there whatever the value.
        const uint32_t vec = sbase + kKvOffVec + st * 1024;
        const int valid = t.lq - qt * kBM;
        const size_t at = static_cast<size_t>(h) * p.total_q + t.q0 + qt * kBM;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = lane + 32 * i;
          const bool in = row < valid;
          cp_async_4(vec + 4 * row, p.nl2t + at + (in ? row : 0), in ? 4u : 0u);
          cp_async_4(vec + 512 + 4 * row, p.nde + at + (in ? row : 0), in ? 4u : 0u);
        }
        cp_async_mbar_arrive(&bars->qd_full[st]);
        __syncwarp();
        mbar_arrive_expect_tx_elect(&bars->qd_full[st], 2 * kTileBytes);
        load_tile(sbase + kKvOffQ + st * 2 * kTileBytes, &tm_q, &bars->qd_full[st], h,
                  t.q0 + qt * kBM);
        load_tile(sbase + kKvOffQ + (st * 2 + 1) * kTileBytes, &tm_do, &bars->qd_full[st], h,
                  t.q0 + qt * kBM);
      }
    }
    if (*abort) {
      for (int i = max(0, ni - kKvBufs); i < ni; ++i)
        mbar_wait_warp(&bars->kv_full[i % kKvBufs], (i / kKvBufs) & 1, abort, err, true);
      for (int i = max(0, S - kQStages); i < S; ++i)
        mbar_wait_warp(&bars->qd_full[i % kQStages], (i / kQStages) & 1, abort, err, true);
    }
  } else if (warp == 9 || warp == 10) {
    // ------------------------------------------------------------------ MMA
    // warp 9: S^T, dP^T of each step once both warpgroups have loaded the
    // previous step's; warp 10: dV += P^T dO and dK += dS^T Q once they have
    // written P^T and dS^T.
    const uint64_t kvdesc0 = sdesc_sw128(sbase + kKvOffK);
    const uint64_t qdesc0 = sdesc_sw128(sbase + kKvOffQ);
    const uint32_t t_dv = tmem + 384, t_dk = tmem + 448;
    const bool is_s = warp == 9;
    int ni = 0, S = 0, done_items = 0;
    bool ok = true;
    for (int nt = 0; ok; ++nt) {
      const int slot = nt & 1;
      if (!mbar_wait_warp(&bars->tile_full[slot], (nt >> 1) & 1, abort, err)) break;
      const KvTile t = bars->tiles[slot];
      if (!t.valid) break;
      if (t.steps > 0) {
        const int kb = ni % kKvBufs;
        if (is_s) {
          ok = mbar_wait_warp(&bars->kv_full[kb], (ni / kKvBufs) & 1, abort, err);
          const uint64_t kd = kvdesc0 + kb * 2 * kTileDesc, vd = kd + kTileDesc;
          for (int s = 0; ok && s < t.steps; ++s) {
            const int g = S + s, st = g % kQStages;
            if (!mbar_wait_warp(&bars->qd_full[st], (g / kQStages) & 1, abort, err) ||
                (g >= 1 && !mbar_wait_warp(&bars->s_read, (g - 1) & 1, abort, err))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t qd = qdesc0 + st * 2 * kTileDesc, dod = qd + kTileDesc;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              umma_ss_elect(tmem, kd + kstep_off(ks), qd + kstep_off(ks), kIdescSS128,
                            ks > 0 ? 1u : 0u);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              umma_ss_elect(tmem + 128, vd + kstep_off(ks), dod + kstep_off(ks), kIdescSS128,
                            ks > 0 ? 1u : 0u);
            umma_commit_elect(&bars->st_full);
            umma_commit_elect(&bars->qd_empty[st]);  // this warp is done with Q / dO
          }
          if (ok) umma_commit_elect(&bars->kv_empty[kb]);
        } else {
          // dV/dK of the previous item must have been read by its epilogue
          if (done_items > 0)
            ok = mbar_wait_warp(&bars->dkv_free, (done_items - 1) & 1, abort, err);
          for (int s = 0; ok && s < t.steps; ++s) {
            const int g = S + s, st = g % kQStages;
            if (!mbar_wait_warp(&bars->ew_done, g & 1, abort, err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // dims 64 half .. of Q and dO: the tiles' swizzle block `half`
            const uint64_t qd = qdesc0 + st * 2 * kTileDesc + t.half * kBlockDesc,
                           dod = qd + kTileDesc;
            // P^T / dS^T of queries 0..127 are 64 consecutive fp16-pair columns
#pragma unroll
            for (int kk = 0; kk < kBM / 16; ++kk)
              umma_ts_elect(t_dv, tmem + 256 + kk * 8, dod + kk * kRows16Desc, kIdescTS,
                            (s > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < kBM / 16; ++kk)
              umma_ts_elect(t_dk, tmem + 320 + kk * 8, qd + kk * kRows16Desc, kIdescTS,
                            (s > 0 || kk > 0) ? 1u : 0u);
            umma_commit_elect(&bars->pds_free);      // P^T / dS^T may be overwritten
            umma_commit_elect(&bars->qd_empty[st]);  // and the stage (its lse / D too)
          }
          if (ok) umma_commit_elect(&bars->dkv_done);
          ++done_items;
        }
        if (!ok) break;
        ++ni;
        S += t.steps;
      }
      if (lane == 0) mbar_arrive(&bars->tile_empty[slot]);
    }
    // every MMA issued by this warp has finished before TMEM is released
    umma_commit_elect(&bars->drain[warp - 9]);
    mbar_wait_warp(&bars->drain[warp - 9], 0, abort, err, true);
  } else {
    // ---------------------------------------- P^T, dS^T (one key / thread)
    const int wg = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_st = tmem + lane_off + 64 * wg, t_dpt = t_st + 128;
    const uint32_t t_pt = tmem + lane_off + 256 + 32 * wg, t_dst = t_pt + 64;
    const uint32_t t_dv = tmem + lane_off + 384 + 32 * wg, t_dk = t_dv + 64;
    int S = 0, done_items = 0;
    bool ok = true;
    for (int nt = 0; ok; ++nt) {
      const int slot = nt & 1;
      if (!mbar_wait_warp(&bars->tile_full[slot], (nt >> 1) & 1, abort, err)) break;
      const KvTile t = bars->tiles[slot];
      if (!t.valid) break;
      const size_t krow = (static_cast<size_t>(t.k0 + t.kt * kBN + r) * p.hkv + t.g) * D +
                          64 * t.half + 32 * wg;
      if (t.steps == 0) {  // no query sees this key tile
        if (r < t.krows) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            reinterpret_cast<uint4 *>(p.dk + krow)[i] = make_uint4(0u, 0u, 0u, 0u);
            reinterpret_cast<uint4 *>(p.dv + krow)[i] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        mbar_arrive(&bars->tile_empty[slot]);
        continue;
      }
      const int jk = t.kt * kBN + r;  // this thread's key
      for (int s = 0; s < t.steps; ++s) {
        const int g = S + s, st = g % kQStages;
        // the lse / D vectors are plain shared-memory stores: wait on their
        // barrier directly, then on the MMAs
        if (!mbar_wait_warp(&bars->qd_full[st], (g / kQStages) & 1, abort, err) ||
            !mbar_wait_warp(&bars->st_full, g & 1, abort, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int qt = t.qt_lo + s % t.nqt;
        // visible query columns of this key among the warpgroup's 64: [c_lo, c_hi)
        const int qb = t.lk - t.lq + qt * kBM + wg * kHalf;  // position of its query 0
        int c_lo = 0, c_hi = min(kHalf, t.lq - qt * kBM - wg * kHalf);
        if (p.causal) c_lo = min(max(jk - qb, 0), kHalf);
        if (p.window > 0) c_hi = min(c_hi, max(jk - qb + p.window, 0));
        const int len = r < t.krows ? max(c_hi - c_lo, 0) : 0;
        // 32-column chunks that some key of the warp does not see whole only
        const int end = c_lo + len;
        const bool mask_a = !__all_sync(0xffffffffu, c_lo <= 0 && end >= 32);
        const bool mask_b = !__all_sync(0xffffffffu, c_lo <= 32 && end >= 64);
        const float *vec =
            reinterpret_cast<const float *>(smem + kKvOffVec + st * 1024) + wg * kHalf;
        uint32_t p16a[16], ds16a[16];
        {
          float sv[32], dp[32];
          tmem_ld32f(t_st, sv);
          tmem_ld32f(t_dpt, dp);
          tmem_wait_ld();
          if (mask_a) mask32(sv, 0, c_lo, len);
          p_ds_col(sv, dp, p.scale_log2, vec, vec + 128, p16a, ds16a);
        }
        float sv[32], dp[32];
        tmem_ld32f(t_st + 32, sv);
        tmem_ld32f(t_dpt + 32, dp);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars->s_read);  // S^T / dP^T of the next step may be computed
        if (mask_b) mask32(sv, 32, c_lo, len);
        uint32_t p16b[16], ds16b[16];
        p_ds_col(sv, dp, p.scale_log2, vec + 32, vec + 128 + 32, p16b, ds16b);
        // dV / dK of step g - 1 have finished reading P^T / dS^T
        if (g >= 1) {
          if (!mbar_wait_warp(&bars->pds_free, (g - 1) & 1, abort, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        tmem_st16(t_pt, p16a);
        tmem_st16(t_dst, ds16a);
        tmem_st16(t_pt + 16, p16b);
        tmem_st16(t_dst + 16, ds16b);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->ew_done);
      }
      if (!ok) break;
      S += t.steps;
      if (!mbar_wait_warp(&bars->dkv_done, done_items & 1, abort, err)) break;
      ++done_items;
      tc_fence_after();
      uint32_t dvv[32], dkv[32];
      tmem_ld32(t_dv, dvv);
      tmem_ld32(t_dk, dkv);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars->dkv_free);
      if (r < t.krows) {
        const float sc = p.scale;
        if constexpr (kV8) {
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const float *x = reinterpret_cast<const float *>(&dvv[16 * i]);
            const float *y = reinterpret_cast<const float *>(&dkv[16 * i]);
            uint32_t wv[8], wk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              wv[e] = pack_bf16x2(x[2 * e], x[2 * e + 1]);
              wk[e] = pack_bf16x2(y[2 * e] * sc, y[2 * e + 1] * sc);
            }
            st_global_v8(p.dv + krow + 16 * i, wv);
            st_global_v8(p.dk + krow + 16 * i, wk);
          }
        } else {
          uint4 *v4 = reinterpret_cast<uint4 *>(p.dv + krow);
          uint4 *k4 = reinterpret_cast<uint4 *>(p.dk + krow);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float *x = reinterpret_cast<const float *>(&dvv[8 * i]);
            const float *y = reinterpret_cast<const float *>(&dkv[8 * i]);
            v4[i] = make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]),
                               pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
            k4[i] = make_uint4(pack_bf16x2(y[0] * sc, y[1] * sc), pack_bf16x2(y[2] * sc, y[3] * sc),
                               pack_bf16x2(y[4] * sc, y[5] * sc), pack_bf16x2(y[6] * sc, y[7] * sc));
          }
        }
      }
      mbar_arrive(&bars->tile_empty[slot]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }
size_t list_bytes(int batch, int64_t total) {  // counter + pairs of one tile list
  return 256 + round256(static_cast<size_t>(total / kBM + batch) * 4);
}

}  // namespace

// Workspace: q16, do16 [total_q, hq, D] fp16; k16, v16 [total_k, hkv, D]
// fp16; nl2t, ndt [hq, total_q] fp32 (+ the exact D nde at D = 128); the
// query-tile and key-tile lists.
size_t backward_workspace_bytes(int batch, int64_t total_q, int64_t total_k, int hq, int hkv,
                                int head_dim) {
  const size_t qb = round256(static_cast<size_t>(total_q) * hq * head_dim * 2);
  const size_t kb = round256(static_cast<size_t>(total_k) * hkv * head_dim * 2);
  const size_t vb = round256(static_cast<size_t>(total_q) * hq * 4);
  return 2 * qb + 2 * kb + (head_dim == 64 ? 2 : 3) * vb + list_bytes(batch, total_q) +
         list_bytes(batch, total_k);
}

namespace {

template <int D, bool kV8>
cudaError_t launch_backward_d(const BackwardLaunch &a, cudaStream_t stream, bool *encode_failed) {
  constexpr int kHalves = TileShape<D>::kHalves;
  uint8_t *ws = static_cast<uint8_t *>(a.workspace);
  const size_t qb = round256(static_cast<size_t>(a.total_q) * a.hq * D * 2);
  const size_t kb = round256(static_cast<size_t>(a.total_k) * a.hkv * D * 2);
  const size_t vb = round256(static_cast<size_t>(a.total_q) * a.hq * 4);
  uint8_t *q16 = ws, *do16 = ws + qb, *k16 = ws + 2 * qb, *v16 = ws + 2 * qb + kb;
  float *nl2t = reinterpret_cast<float *>(ws + 2 * qb + 2 * kb);
  float *ndt = reinterpret_cast<float *>(ws + 2 * qb + 2 * kb + vb);
  // exact D: in place of the forward's at D = 64 (one item per row and head);
  // its own array at D = 128, where both halves of a row read the forward's
  float *nde = D == 64 ? ndt : reinterpret_cast<float *>(ws + 2 * qb + 2 * kb + 2 * vb);
  uint8_t *qlist = ws + 2 * qb + 2 * kb + (D == 64 ? 2 : 3) * vb;
  uint8_t *klist = qlist + list_bytes(a.batch, a.total_q);

  cudaError_t e;
  if (a.total_q > 0) {
    const int64_t n = a.total_q * a.hq * (D / 8);
    const int64_t blocks = (n + 255) / 256;
    bwd_prep_q_kernel<D><<<static_cast<unsigned>(blocks < 8192 ? blocks : 8192), 256, 0,
                           stream>>>(
        static_cast<const uint4 *>(a.q), static_cast<const uint4 *>(a.dout),
        static_cast<const uint4 *>(a.out), a.lse, a.total_q, a.hq, reinterpret_cast<uint4 *>(q16),
        reinterpret_cast<uint4 *>(do16), nl2t, ndt);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (a.total_k > 0) {
    const int64_t n8 = a.total_k * a.hkv * (D / 8);
    const int64_t blocks = (n8 + 255) / 256;
    bwd_prep_kv_kernel<<<static_cast<unsigned>(blocks < 8192 ? blocks : 8192), 256, 0, stream>>>(
        static_cast<const uint4 *>(a.k), static_cast<const uint4 *>(a.v),
        reinterpret_cast<uint4 *>(k16), reinterpret_cast<uint4 *>(v16), n8);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const int max_qtiles = (a.max_seqlen_q + kBM - 1) / kBM;
  const int max_ktiles = (a.max_seqlen_k + kBN - 1) / kBN;
  BwdParams p;
  p.cu_q = a.cu_q;
  p.cu_k = a.cu_k;
  p.batch = a.batch;
  p.hq = a.hq;
  p.hkv = a.hkv;
  p.group = a.hq / a.hkv;
  p.causal = a.causal ? 1 : 0;
  p.window = a.window;
  p.total_q = static_cast<int>(a.total_q);
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.nl2t = nl2t;
  p.ndt = ndt;
  p.nde = nde;
  p.q_pairs = reinterpret_cast<const unsigned *>(qlist + 256);
  p.num_q_pairs = reinterpret_cast<const int *>(qlist + 4);
  p.q_counter = reinterpret_cast<unsigned *>(qlist);
  p.k_counter = reinterpret_cast<unsigned *>(klist);
  p.k_pairs = reinterpret_cast<const unsigned *>(klist + 256);
  p.num_k_pairs = reinterpret_cast<const int *>(klist + 4);
  p.dq = static_cast<__nv_bfloat16 *>(a.dq);
  p.dk = static_cast<__nv_bfloat16 *>(a.dk);
  p.dv = static_cast<__nv_bfloat16 *>(a.dv);
  p.stall_ns = g_bwd_stall_ns.load();
  if ((e = launch_tile_list(a.cu_q, a.batch, max_qtiles, reinterpret_cast<unsigned *>(qlist + 256),
                            reinterpret_cast<int *>(qlist + 4), reinterpret_cast<unsigned *>(qlist),
                            stream)) != cudaSuccess)
    return e;
  if ((e = launch_tile_list(a.cu_k, a.batch, max_ktiles, reinterpret_cast<unsigned *>(klist + 256),
                            reinterpret_cast<int *>(klist + 4), reinterpret_cast<unsigned *>(klist),
                            stream)) != cudaSuccess)
    return e;

  EncodeTiledFn fn = get_encode_fn();
  CUtensorMap tq, tdo, tk, tv;
  const CUtensorMapDataType f16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  // with no keys (or queries) nothing reads those maps; they then point at q16
  const void *kbase = a.total_k > 0 ? static_cast<const void *>(k16) : q16;
  const void *vbase = a.total_k > 0 ? static_cast<const void *>(v16) : q16;
  if (fn == nullptr || !encode_rows_heads(fn, &tq, q16, a.total_q, a.hq, f16, D) ||
      !encode_rows_heads(fn, &tdo, do16, a.total_q, a.hq, f16, D) ||
      !encode_rows_heads(fn, &tk, kbase, a.total_k, a.hkv, f16, D) ||
      !encode_rows_heads(fn, &tv, vbase, a.total_k, a.hkv, f16, D)) {
    *encode_failed = true;
    return cudaErrorInvalidValue;
  }
  constexpr int kDqSmem = DqCfg<D>::kSmem, kKvSmem = KvCfg<D>::kSmem;
  if ((e = cudaFuncSetAttribute(bwd_dq_kernel<D, kV8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kDqSmem)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(bwd_dkdv_kernel<D, kV8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kKvSmem)) != cudaSuccess)
    return e;
  if (a.total_q > 0) {
    const int64_t items = (a.total_q / kBM + a.batch) * a.hq * kHalves;
    const int64_t grid = items < sm_count() ? items : sm_count();
    bwd_dq_kernel<D, kV8><<<static_cast<unsigned>(grid), kDqThreads, kDqSmem, stream>>>(
        tq, tdo, tk, tv, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const bool dsink = a.sinks != nullptr && a.dsinks != nullptr;
  if (dsink) {  // after dQ: D is exact by now
    bwd_dsink_kernel<<<a.hq, 256, 0, stream>>>(a.sinks, nl2t, nde, a.total_q, a.dsinks);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (a.total_k > 0) {
    const int64_t items = (a.total_k / kBN + a.batch) * a.hkv * kHalves;
    const int64_t grid = items < sm_count() ? items : sm_count();
    // overlaps the sink gradient (programmatic dependent launch); everything
    // it reads was written before that kernel started
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kKvThreads);
    cfg.dynamicSmemBytes = kKvSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dsink ? 1 : 0;
    if ((e = cudaLaunchKernelEx(&cfg, bwd_dkdv_kernel<D, kV8>, tq, tdo, tk, tv, p)) != cudaSuccess)
      return e;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_backward(const BackwardLaunch &a, cudaStream_t stream, bool *encode_failed) {
  *encode_failed = false;
  if (a.batch == 0) return cudaSuccess;
  const bool v8 = ((reinterpret_cast<uintptr_t>(a.dq) | reinterpret_cast<uintptr_t>(a.dk) |
                   reinterpret_cast<uintptr_t>(a.dv)) & 31u) == 0;
  if (a.head_dim == 128)
    return v8 ? launch_backward_d<128, true>(a, stream, encode_failed)
              : launch_backward_d<128, false>(a, stream, encode_failed);
  return v8 ? launch_backward_d<64, true>(a, stream, encode_failed)
            : launch_backward_d<64, false>(a, stream, encode_failed);
}

cudaError_t backward_set_stall(uint64_t ns) {
  g_bwd_stall_ns.store(ns);
  return cudaSuccess;
}

cudaError_t backward_read_error(cudaStream_t stream, int *code) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(code, g_backward_error, sizeof(int));
  const int zero = 0;
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_backward_error, &zero, sizeof(int));
  return e;
}

}  // namespace sinkattn
