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
// One CTA = 128 query rows x NT query heads (NT = 2 heads of one KV group
// when the group size is even, else 1); every K/V tile is shared by the NT
// tiles. Warps (NT = 2):
//   warps 0-3, 4-7  softmax warpgroup t: thread r owns row r of tile t (TMEM lane r)
//   warp 8          TMA producer: tiles, both Q tiles once, then K_j into a 3-stage ring
//   warp 9          P V issuer and TMEM owner
//   warp 10         Q K^T issuer
//   warp 11         TMA producer of V_j (its own 3-stage ring)
// (NT = 1: one softmax warpgroup, warps 4-7 in the same roles.) A K stage is
// released once the tile's Q K^T has read it and a V stage once its P V has,
// so K loads never wait for P V. setmaxnreg moves registers from warps 8-11
// (88 each) to the two softmax warpgroups (208 each).
// TMEM (512 columns): O_t at [384 + D t, ...) and score buffers in
// [0, 384). NT = 2: three 128-column S buffers shared round-robin by the work
// items k = NT j + t (KV tile j, query tile t); P_k (fp16 pairs) overwrites
// the first 64 columns of its S buffer once S_k has been read, and feeds P V
// straight from TMEM; Q K^T runs up to two items ahead of the softmax.
// NT = 1: two S buffers and two separate 64-column P buffers at 256; an S
// buffer is released as soon as the softmax has loaded it, so the next
// scores are computed while the softmax works on the current ones.
// Softmax: one read of the 128 scores of a row from TMEM, a range mask on
// boundary tiles only, tree reductions (3-input max), packed f32x2 arithmetic
// and hardware ex2. The running maximum is only
// moved (and O, d rescaled) when it grows by more than 8 in log2 units; the
// final division uses the same reference maximum, so the result is unchanged
// while most tiles skip the O round trip.
#include <math.h>

#include <algorithm>
#include <atomic>
#include <type_traits>
#include <mutex>

#include "launch.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace sinkattn {
namespace {

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per KV tile
constexpr int kMaxStages = 3;                    // K/V ring depth at head_dim 64 (2 at 128)
constexpr int kBlockBytes = kBM * 64 * 2;        // 16 KB: 128 rows x 64 elements, one swizzle block
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// NT query heads per item (2 when the group size is even), head dimension D:
// 64 (NT 1 or 2) or 128 (NT 1). A 128-row tile of one head is D / 64
// blocks of 128 rows x 128 bytes, each loaded by one TMA box with 128-byte
// swizzle; at D = 128 the K and V rings have two stages so that two Q
// buffers and the rings fit in shared memory, and O (128 columns) fills TMEM
// beside the score buffers.
template <int NT, int D>
struct Cfg {
  // NT = 2: three full warpgroups, so setmaxnreg can move registers from the
  // producer/MMA warpgroup to the two softmax warpgroups.
  static constexpr int kThreads = NT * 128 + 128;
  static constexpr int kProducerWarp = NT * 4;   // tiles, Q and K loads
  static constexpr int kMmaWarp = NT * 4 + 1;    // P V issuer, TMEM owner
  static constexpr int kQkWarp = NT * 4 + 2;     // Q K^T issuer
  static constexpr int kVWarp = NT * 4 + 3;      // V loads
  // One head per item at head_dim 64: two CTAs per SM, each with half the
  // TMEM (256 columns) and half the registers.
  static constexpr bool kDual = NT == 1 && D == 64;
  static constexpr int kMinBlocks = kDual ? 2 : 1;
  // Score buffers. Two heads per item: three 128-column S buffers used
  // round-robin by the items, P written over its S, O_t at 384 + 64 t. One
  // head per item: kSBufs S buffers and as many separate 64-column P buffers,
  // so an S buffer is free as soon as the softmax has loaded it (two of each
  // at head_dim 128, one of each in a dual CTA), then O.
  static constexpr bool kSplitP = NT == 1;
  static constexpr int kSBufs = kSplitP ? (kDual ? 1 : 2) : 3;
  static constexpr uint32_t kTmemP = kSplitP ? kSBufs * 128 : 0;
  static constexpr uint32_t kTmemO = kSplitP ? kTmemP + kSBufs * 64 : 384;
  static constexpr uint32_t kTmemCols = kDual ? 256 : 512;
  static constexpr int kTile = kBM * D * 2;                        // one 128-row tile of one head
  static constexpr int kStages = D == 64 && !kDual ? 3 : 2;
  static constexpr int kOffQ = 0;                                  // 2 buffers x NT tiles
  static constexpr int kOffK = kOffQ + 2 * NT * kTile;
  static constexpr int kOffV = kOffK + kStages * kTile;
  static constexpr int kOffBar = kOffV + kStages * kTile;
  static constexpr int kOffPend = kOffBar + 1024;  // 16 B per softmax thread: deferred epilogue
  static constexpr int kOffPendVs = kOffPend + NT * 128 * 16;  // + its value scale (4 B)
  static constexpr int kSmemBytes = kOffPendVs + NT * 128 * 4 + 1024;  // + alignment slack
};

// Register split of the NT = 2 kernel (setmaxnreg): 168 registers a thread at
// launch (the ptxas limit for 384 threads), then 88 for the producer / MMA
// warpgroup and 208 for each softmax warpgroup (72 / 216 made the producer
// path spill: window-128 prefill 6% slower).
constexpr int kLaunchRegs2 = 168;
constexpr int kRegsOther2 = 88;
constexpr int kRegsSoftmax2 = 208;
static_assert(kRegsOther2 * 128 + kRegsSoftmax2 * 256 <= kLaunchRegs2 * Cfg<2, 64>::kThreads,
              "register split must fit the registers the block is launched with");
// Dual CTAs (one head per item, head_dim 64, two CTAs per SM): 128 registers
// a thread at launch, then 72 for the producer / MMA warps (64 made them
// spill) and 184 for the softmax warpgroup.
constexpr int kLaunchRegsD = 128;
constexpr int kRegsOtherD = 72;
constexpr int kRegsSoftmaxD = 184;
static_assert(kRegsOtherD * 128 + kRegsSoftmaxD * 128 <= kLaunchRegsD * Cfg<1, 64>::kThreads,
              "register split must fit the registers the block is launched with");

constexpr uint32_t kIdescQK = idesc_f32acc(kBM, kBN, /*bf16=*/true, false, false);
constexpr uint32_t kIdescPV = idesc_f32acc(kBM, 64, /*bf16=*/false, false, true);  // per 64 dims

__device__ int g_prefill_error;

struct Params {
  const int32_t *cu_q, *cu_k;
  int batch, hq, group, causal, window, max_qtiles;
  const float *sinks;
  float scale_log2;
  __nv_bfloat16 *out;
  float *lse;
  unsigned int *work_counter;  // zeroed by build_worklist_kernel
  const unsigned *work_pairs;  // longest-first (sequence, query tile) list, packed b << 16 | qt
  const int *num_pairs;        // its length
  // Split-KV: with num_splits > 1 every (tile, heads) item is cut into that
  // many key ranges; split s writes its normalised partial output and lse to
  // part_o [s][total_q][hq][D] / part_lse [s][total_q][hq] (fp32) instead of
  // out/lse, and only split 0 starts from the sink.
  int num_splits, total_q;
  float *part_o, *part_lse;
  // Per-KV-head value scales of an fp8 cache (NULL: 1). Key j of KV head g
  // stands for k_scale[g] * K_j: k_scale multiplies the softmax scale, and
  // v_scale the normalised output (it is linear in V).
  const float *k_scale, *v_scale;
  // Testing hook (0: off): the softmax warps' first score wait of each CTA is
  // preceded by a wait of at most stall_ns on a barrier that nothing
  // completes, so that every CTA takes its timeout path.
  uint64_t stall_ns;
};

// One unit of work: 128 query rows of sequence b for the NT heads h0...
struct Tile {
  int valid;  // 0: no more work
  int h0, b, qt, q0, lq, k0, lk, rows, kvh, p_min, p_max, kt_lo, n, split;
  float sink_log2[2];  // initial running maximum of head h0 + t (log2 units; -inf: none)
};

struct Barriers {
  uint64_t q_full[2], q_empty[2];       // double-buffered Q tiles
  uint64_t k_full[kMaxStages], k_empty[kMaxStages];  // K ring: freed once Q K^T has read it
  uint64_t v_full[kMaxStages], v_empty[kMaxStages];  // V ring: freed once P V has read it
  uint64_t s_full[3];                   // S of item k in buffer k % kSBufs
  uint64_t s_read[2];                   // separate P: the softmax has loaded S (buffer free)
  uint64_t p_full[3];                   // P of item k written (buffer k % kSBufs)
  uint64_t pv_done[3];                  // P V of that item has completed
  uint64_t o_done[2];                   // one phase per P V into O_t
  uint64_t o_free[2];                   // one phase per tile with keys: epilogue has read O_t
  uint64_t tile_full[2], tile_empty[2]; // tile descriptor ring
  uint64_t drain[2];
  uint64_t never;                       // testing hook: a barrier nothing completes
  uint32_t tmem_base;
  int abort;
  Tile tiles[2];
};
static_assert(sizeof(Barriers) <= 1024, "control block");

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float row_max32(const float (&sv)[32]) {
  float m[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) m[i] = max3(sv[8 * i], sv[8 * i + 1], sv[8 * i + 2]);
#pragma unroll
  for (int i = 0; i < 4; ++i) m[i] = max3(m[i], sv[8 * i + 3], sv[8 * i + 4]);
#pragma unroll
  for (int i = 0; i < 4; ++i) m[i] = max3(m[i], sv[8 * i + 5], sv[8 * i + 6]);
  return max3(max3(m[0], m[1], m[2]), m[3], max3(sv[7], sv[15], max3(sv[23], sv[31], m[0])));
}

// 32 scores -> 2^(x c - m) as 16 fp16 pairs into pk[off..off+16); row sums into acc.
// Exponentials on the special-function unit (ex2(-inf) = 0 for masked keys),
// which retires about 30 results per clock per SM on GB300. Moving a share of
// them to an FMA-pipe polynomial made this kernel slower: the extra
// instructions lengthen the softmax, which sits on each tile's dependency
// chain (Q K^T -> softmax -> P V -> the next Q K^T into the same buffer).
__device__ __forceinline__ void exp32(const float (&sv)[32], float2 c2, float2 nb2,
                                      float2 (&acc)[4], uint32_t (&pk)[32], int off) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float2 a = __ffma2_rn(make_float2(sv[2 * i], sv[2 * i + 1]), c2, nb2);
    const float2 e = make_float2(fast_exp2(a.x), fast_exp2(a.y));
    acc[i & 3] = __fadd2_rn(acc[i & 3], e);
    pk[off + i] = pack_f16x2(e.x, e.y);
  }
}

// Work index w -> tile. Splits are outermost (items that run at the same time
// share a key range, which keeps it in L2); within a split, list entry
// (w / groups) gives (sequence, query tile) and w % groups the head group.
// n = 0 for a tile that sees no key (in this split).
__device__ __forceinline__ void decode_work(const Params &p, int NT, int npairs, int w, Tile &t) {
  const int groups = p.hq / NT;
  const int split = w / (npairs * groups);
  w -= split * npairs * groups;
  const unsigned e = p.work_pairs[w / groups];
  const int b = static_cast<int>(e >> 16), qt = static_cast<int>(e & 0xffffu);
  const int q0 = p.cu_q[b], lq = p.cu_q[b + 1] - q0;
  t.valid = 1;
  t.split = split;
  t.h0 = (w % groups) * NT;
  t.b = b;
  t.qt = qt;
  t.q0 = q0;
  t.lq = lq;
  t.k0 = p.cu_k[b];
  t.lk = p.cu_k[b + 1] - t.k0;
  t.rows = min(kBM, lq - qt * kBM);
  t.kvh = t.h0 / p.group;
  t.p_min = t.lk - lq + qt * kBM;  // position of the tile's first query
  t.p_max = t.p_min + t.rows - 1;
  int key_hi = t.lk, key_lo = 0;
  if (p.causal) key_hi = min(key_hi, t.p_max + 1);
  if (p.window > 0) key_lo = max(0, t.p_min - p.window + 1);
  t.kt_lo = key_lo / kBN;
  t.n = key_hi > key_lo ? (key_hi + kBN - 1) / kBN - t.kt_lo : 0;
  // the sink enters split 0 only; read here, off the softmax warps' path
  for (int i = 0; i < 2; ++i)
    t.sink_log2[i] = p.sinks != nullptr && split == 0 && i < NT ? p.sinks[t.h0 + i] * kLog2e
                                                                : -INFINITY;
  if (p.num_splits > 1) {  // this split's share of the key tiles
    const int lo = static_cast<int>(static_cast<int64_t>(t.n) * split / p.num_splits);
    const int hi = static_cast<int>(static_cast<int64_t>(t.n) * (split + 1) / p.num_splits);
    t.kt_lo += lo;
    t.n = hi - lo;
  }
}

// One block: the list of non-empty (sequence b, query tile qt) pairs, ordered
// by qt descending (the tiles with the most keys first under a causal mask),
// and the zeroed work counter. Levels (one per qt) are counted with a
// histogram of tiles per sequence, offset by a scan, then filled.
constexpr int kMaxLevels = 4096;  // longer sequences: pairs in sequence order

// Exclusive scan of one int per thread across a block of blockDim.x (a
// multiple of 32, at most 1024) threads; returns this thread's prefix and the
// block total.
__device__ __forceinline__ int block_exclusive_scan(int x, int *total) {
  __shared__ int warp_sums[32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int nw = blockDim.x >> 5;
    int v = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    warp_sums[lane] = v;  // inclusive prefix over warps
  }
  __syncthreads();
  const int warp_off = wid > 0 ? warp_sums[wid - 1] : 0;
  *total = warp_sums[(blockDim.x >> 5) - 1];
  return warp_off + incl - x;
}

// One block: the list of non-empty (sequence b, query tile qt) pairs, ordered
// by qt descending (the tiles with the most keys first under a causal mask),
// and the zeroed work counter. Levels (one per qt) are counted, offset by a
// block scan, then filled. The host passes an upper bound on every length: a
// sequence longer than max_qtiles tiles is cut to that bound and recorded in
// the device error word (code 3).
__global__ void __launch_bounds__(1024) build_worklist_kernel(const int32_t *cu_q, int batch,
                                                               int max_qtiles, unsigned *pairs,
                                                               int *num_pairs,
                                                               unsigned int *counter) {
  __shared__ int level_start[kMaxLevels];
  __shared__ int level_fill[kMaxLevels];
  const int tid = threadIdx.x;
  if (tid == 0) *counter = 0u;
  if (max_qtiles <= kMaxLevels) {
    // level z holds qt = max_qtiles - 1 - z; count tiles per level
    for (int z = tid; z < max_qtiles; z += blockDim.x) {
      level_start[z] = 0;
      level_fill[z] = 0;
    }
    __syncthreads();
    for (int b = tid; b < batch; b += blockDim.x) {
      const int full = (cu_q[b + 1] - cu_q[b] + kBM - 1) / kBM;
      if (full > max_qtiles) atomicExch(&g_prefill_error, kErrBadLength);
      const int nq = min(full, max_qtiles);
      for (int qt = 0; qt < nq; ++qt) atomicAdd(&level_start[max_qtiles - 1 - qt], 1);
    }
    __syncthreads();
    // exclusive scan over the levels: each thread owns a run of `per` levels
    const int per = (max_qtiles + blockDim.x - 1) / blockDim.x;
    const int z0 = min(tid * per, max_qtiles), z1 = min(z0 + per, max_qtiles);
    int local = 0;
    for (int z = z0; z < z1; ++z) local += level_start[z];
    int total = 0;
    int run = block_exclusive_scan(local, &total);
    for (int z = z0; z < z1; ++z) {
      const int c = level_start[z];
      level_start[z] = run;
      run += c;
    }
    if (tid == 0) *num_pairs = total;
    __syncthreads();
    for (int b = tid; b < batch; b += blockDim.x) {
      const int nq = min((cu_q[b + 1] - cu_q[b] + kBM - 1) / kBM, max_qtiles);
      for (int qt = 0; qt < nq; ++qt) {
        const int z = max_qtiles - 1 - qt;
        pairs[level_start[z] + atomicAdd(&level_fill[z], 1)] =
            (static_cast<unsigned>(b) << 16) | static_cast<unsigned>(qt);
      }
    }
  } else if (tid == 0) {
    int run = 0;
    for (int b = 0; b < batch; ++b) {
      const int full = (cu_q[b + 1] - cu_q[b] + kBM - 1) / kBM;
      if (full > max_qtiles) atomicExch(&g_prefill_error, kErrBadLength);
      const int nq = min(full, max_qtiles);
      for (int qt = nq - 1; qt >= 0; --qt)
        pairs[run++] = (static_cast<unsigned>(b) << 16) | static_cast<unsigned>(qt);
    }
    *num_pairs = run;
  }
}

// Persistent: one CTA per SM takes tiles from a global counter until the list
// is exhausted. Every role keeps running counters (S buffer items, K/V stages,
// Q buffers, tiles) across tiles, so the next tile's loads and Q K^T overlap
// the current tile's softmax and epilogue.
// kV8: out (and part_o) start on 32-byte boundaries, and each output row is
// stored with 32-byte stores (whole sectors, half the store instructions);
// otherwise with 16-byte ones.
template <int NT, int D, bool kV8>
__global__ void __launch_bounds__(Cfg<NT, D>::kThreads, Cfg<NT, D>::kMinBlocks)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const Params p) {
  using C = Cfg<NT, D>;
  constexpr int kStages = C::kStages;
  constexpr int kTileBytes = C::kTile;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (sbase - raw);
  Barriers *bars = reinterpret_cast<Barriers *>(smem + C::kOffBar);
  volatile int *abort = &bars->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
      mbar_init(&bars->o_done[i], 1);
      mbar_init(&bars->o_free[i], kBM);
      mbar_init(&bars->tile_full[i], 1);
      mbar_init(&bars->tile_empty[i], NT * kBM + 3);
      mbar_init(&bars->drain[i], 1);
    }
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int i = 0; i < 3; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], kBM);
      mbar_init(&bars->pv_done[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_read[i], kBM);
    }
    mbar_init(&bars->never, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(&bars->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp >= C::kProducerWarp) {
    if constexpr (NT == 2)
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther2));
    else if constexpr (C::kDual)
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOtherD));
    if (warp == C::kProducerWarp) {
      // ---------------------------------------------------------- producer
      // Fetches tiles, publishes them in the 2-slot ring, and streams each
      // tile's Q (double-buffered) and K tiles (3-stage ring; V has its own
      // ring and warp, so a K load never waits for P V to free a V stage).
      // The whole warp runs the loop; lane 0 fetches and publishes, one
      // elected lane issues each copy.
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      // one tile = D / 64 boxes of 64 elements, into consecutive 16 KB blocks
      auto load_tile = [&](uint32_t dst, const CUtensorMap *map, uint64_t *bar, int head, int row) {
#pragma unroll
        for (int blk = 0; blk < D / 64; ++blk)
          tma_load_3d_elect(dst + blk * kBlockBytes, map, bar, blk * 64, head, row);
      };
      int J = 0;  // K/V stage uses so far
      int q_loads = 0;
      const int npairs = *p.num_pairs;
      const int num_work = npairs * (p.hq / NT) * p.num_splits;
      for (int nt = 0;; ++nt) {
        const int slot = nt & 1;
        if (nt >= 2 && !mbar_wait_warp(&bars->tile_empty[slot], ((nt >> 1) - 1) & 1, abort,
                                       &g_prefill_error))
          break;
        if (lane == 0) {
          Tile t;
          t.valid = 0;
          const int w = static_cast<int>(atomicAdd(p.work_counter, 1u));
          if (w < num_work) decode_work(p, NT, npairs, w, t);
          bars->tiles[slot] = t;
          mbar_arrive(&bars->tile_full[slot]);
        }
        __syncwarp();
        const Tile t = bars->tiles[slot];
        if (!t.valid) break;
        const int qb = nt & 1;
        if (nt >= 2 && !mbar_wait_warp(&bars->q_empty[qb], ((nt >> 1) - 1) & 1, abort,
                                       &g_prefill_error))
          break;
        mbar_arrive_expect_tx_elect(&bars->q_full[qb], NT * kTileBytes);
        ++q_loads;
        for (int i = 0; i < NT; ++i)
          load_tile(sbase + C::kOffQ + (qb * NT + i) * kTileBytes, &tm_q, &bars->q_full[qb],
                    t.h0 + i, t.q0 + t.qt * kBM);
        bool ok = true;
        for (int j = 0; j < t.n; ++j, ++J) {
          const int st = J % kStages;
          if (J >= kStages && !mbar_wait_warp(&bars->k_empty[st], ((J / kStages) - 1) & 1, abort,
                                              &g_prefill_error)) {
            ok = false;
            break;
          }
          const int row = t.k0 + (t.kt_lo + j) * kBN;
          mbar_arrive_expect_tx_elect(&bars->k_full[st], kTileBytes);
          load_tile(sbase + C::kOffK + st * kTileBytes, &tm_k, &bars->k_full[st], t.kvh, row);
        }
        if (!ok) break;
      }
      if (*abort) {
        // Copies already issued still land in this CTA's shared memory: wait
        // for the last ones of each ring (bounded) before the CTA may exit.
        for (int i = max(0, q_loads - 2); i < q_loads; ++i)
          mbar_wait_warp(&bars->q_full[i & 1], (i >> 1) & 1, abort, &g_prefill_error, true);
        for (int i = max(0, J - kStages); i < J; ++i)
          mbar_wait_warp(&bars->k_full[i % kStages], (i / kStages) & 1, abort, &g_prefill_error,
                         true);
      }
    } else if (warp == C::kVWarp) {
      // --------------------------------------------------------- V producer
      // Follows the published tiles and streams their V tiles into the V ring.
      // V may still be being converted to fp16 by the grid launched before
      // this one: wait for it here, the kernel's only use of V.
      asm volatile("griddepcontrol.wait;" ::: "memory");
      tma_prefetch_desc(&tm_v);
      int J = 0;
      for (int nt = 0;; ++nt) {
        const int slot = nt & 1;
        if (!mbar_wait_warp(&bars->tile_full[slot], (nt >> 1) & 1, abort, &g_prefill_error))
          break;
        const Tile t = bars->tiles[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->tile_empty[slot]);
        if (!t.valid) break;
        bool ok = true;
        for (int j = 0; j < t.n; ++j, ++J) {
          const int st = J % kStages;
          if (J >= kStages && !mbar_wait_warp(&bars->v_empty[st], ((J / kStages) - 1) & 1, abort,
                                              &g_prefill_error)) {
            ok = false;
            break;
          }
          const int row = t.k0 + (t.kt_lo + j) * kBN;
          mbar_arrive_expect_tx_elect(&bars->v_full[st], kTileBytes);
#pragma unroll
          for (int blk = 0; blk < D / 64; ++blk)
            tma_load_3d_elect(sbase + C::kOffV + st * kTileBytes + blk * kBlockBytes, &tm_v,
                              &bars->v_full[st], blk * 64, t.kvh, row);
        }
        if (!ok) break;
      }
      if (*abort) {
        for (int i = max(0, J - kStages); i < J; ++i)
          mbar_wait_warp(&bars->v_full[i % kStages], (i / kStages) & 1, abort, &g_prefill_error,
                         true);
      }
    } else if (warp == C::kMmaWarp || warp == C::kQkWarp) {
      // ------------------------------------------------------- MMA issuers
      // Work items k = NT j + t of a tile (KV tile j, query tile t), counted
      // globally across tiles (K); item K uses score buffer K % kSBufs. With
      // P written over S (two heads), the Q K^T warp issues QK(K) once PV(K -
      // 3) has completed, so Q K^T runs up to two items ahead of the softmax;
      // with separate P buffers (one head), once the softmax has loaded the
      // scores of item K - 2, so the next scores are computed while the
      // softmax works on the current ones. The P V warp issues PV(K) once the
      // softmax has written P. Each warp runs its loop whole (uniform
      // operands); one elected lane issues each MMA and commit.
      constexpr uint64_t kTileDesc = kTileBytes >> 4;   // one tile, in descriptor address units
      constexpr uint64_t kBlockDesc = kBlockBytes >> 4;  // one 64-element block of a tile
      const int role = warp == C::kMmaWarp ? 0 : 1;
      const uint64_t qdesc0 = sdesc_sw128(sbase + C::kOffQ);
      const uint64_t kdesc0 = sdesc_sw128(sbase + C::kOffK);
      const uint64_t vdesc0 = sdesc_sw128(sbase + C::kOffV);
      int K = 0, J = 0;
      int o_free_waits[2] = {0, 0};  // P V warp: o_free phases consumed per tile slot t
      bool o_used = false;           // an earlier tile wrote O (had keys)
      for (int nt = 0;; ++nt) {
        const int slot = nt & 1;
        if (!mbar_wait_warp(&bars->tile_full[slot], (nt >> 1) & 1, abort, &g_prefill_error))
          break;
        const Tile t = bars->tiles[slot];
        if (!t.valid) break;
        const int items = NT * t.n;
        bool ok = true;
        if (role == 1) {
          const int qb = nt & 1;
          ok = mbar_wait_warp(&bars->q_full[qb], (nt >> 1) & 1, abort, &g_prefill_error);
          for (int k = 0; ok && k < items; ++k) {
            const int tt = k % NT, jj = k / NT, KK = K + k, b = KK % C::kSBufs;
            const bool free_ok =
                C::kSplitP
                    ? (KK < C::kSBufs ||
                       mbar_wait_warp(&bars->s_read[b], ((KK - C::kSBufs) / C::kSBufs) & 1,
                                      abort, &g_prefill_error))
                    : (KK < 3 || mbar_wait_warp(&bars->pv_done[b], ((KK - 3) / 3) & 1, abort,
                                                &g_prefill_error));
            if (!free_ok) {
              ok = false;
              break;
            }
            const int Jc = J + jj;
            if (tt == 0 && !mbar_wait_warp(&bars->k_full[Jc % kStages], (Jc / kStages) & 1, abort,
                                           &g_prefill_error)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t qd = qdesc0 + (qb * NT + tt) * kTileDesc;
            const uint64_t kd = kdesc0 + (Jc % kStages) * kTileDesc;
            const uint32_t sbuf = tmem + b * kBN;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {  // k-step ks: block ks / 4, 32-byte step ks % 4
              const uint64_t off = (ks >> 2) * kBlockDesc + 2 * (ks & 3);
              umma_ss_elect(sbuf, qd + off, kd + off, kIdescQK, ks > 0 ? 1u : 0u);
            }
            umma_commit_elect(&bars->s_full[b]);
            // the K stage is free once the tile's last Q K^T has read it
            if (tt == NT - 1) umma_commit_elect(&bars->k_empty[Jc % kStages]);
          }
          if (ok) umma_commit_elect(&bars->q_empty[qb]);  // Q buffer free once these QK finish
        } else {
          for (int k = 0; ok && k < items; ++k) {
            const int tt = k % NT, jj = k / NT, KK = K + k, b = KK % C::kSBufs, Jc = J + jj;
            // the first P V of a tile into O_t waits until the epilogue of the
            // last tile that used O_t (same softmax warpgroup) has read it; only
            // tiles with keys use O_t and signal o_free, so the phases pair up
            if (jj == 0 && o_used && !mbar_wait_warp(&bars->o_free[tt], o_free_waits[tt] & 1,
                                                     abort, &g_prefill_error)) {
              ok = false;
              break;
            }
            if (jj == 0 && o_used) ++o_free_waits[tt];
            if (tt == 0 && !mbar_wait_warp(&bars->v_full[Jc % kStages], (Jc / kStages) & 1, abort,
                                           &g_prefill_error)) {
              ok = false;
              break;
            }
            if (!mbar_wait_warp(&bars->p_full[b], (KK / C::kSBufs) & 1, abort, &g_prefill_error)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t vd = vdesc0 + (Jc % kStages) * kTileDesc;
            const uint32_t pbuf = tmem + (C::kSplitP ? C::kTmemP + b * 64 : b * kBN);
            const uint32_t obuf = tmem + C::kTmemO + tt * D;
#pragma unroll
            for (int hb = 0; hb < D / 64; ++hb)  // O columns of dims 64 hb.. from V block hb
#pragma unroll
              for (int kk = 0; kk < kBN / 16; ++kk)
                umma_ts_elect(obuf + hb * 64, pbuf + kk * 8,
                              vd + hb * kBlockDesc + kk * (16 * 128 / 16), kIdescPV,
                              (jj > 0 || kk > 0) ? 1u : 0u);
            umma_commit_elect(&bars->o_done[tt]);
            umma_commit_elect(&bars->pv_done[b]);
            // the V stage is free after the tile's last P V
            if (tt == NT - 1) umma_commit_elect(&bars->v_empty[Jc % kStages]);
          }
        }
        if (!ok) break;
        if (t.n > 0) o_used = true;
        if (lane == 0) mbar_arrive(&bars->tile_empty[slot]);
        K += items;
        J += t.n;
      }
      // every MMA issued by this warp has finished before TMEM is released
      umma_commit_elect(&bars->drain[role]);
      mbar_wait_warp(&bars->drain[role], 0, abort, &g_prefill_error, true);
    }
  } else {
    if constexpr (NT == 2)
      asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax2));
    else if constexpr (C::kDual)
      asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmaxD));
    // -------------------------------------------------------------- softmax
    const int t = warp >> 2;          // which query tile (head h0 + t)
    const int r = threadIdx.x & 127;  // row within the tile == TMEM lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t o_addr = lane_addr + C::kTmemO + t * D;
    int K = 0;        // items of earlier tiles
    // Within an item the softmax waits for the previous P V into O_t only
    // where it must rescale O_t, and on the item's last tile; the epilogue
    // waits for the item's last P V. The waits name the phase by index:
    // o_base = P V products into O_t before this item, o_pend = index of the
    // pending item's last one. A parity wait is unambiguous when the barrier
    // is at most one phase from the one waited for:
    // - at tile j, P V(t, j - 2) is complete: with P over S (two heads), S of
    //   item k is in only after P V(k - 3) has completed; with separate P
    //   buffers (one head), P of item k is written only after P V(k - kSBufs)
    //   has completed, kSBufs <= 2; and a commit completes only after every
    //   earlier product of its issuing thread. P V(t, j) is not yet issued;
    // - the epilogue can run without a later score wait in between (after an
    //   item without keys, or at the end), so the wait on the item's last
    //   tile (for P V(t, n - 2)) is what bounds it from below; the next P V
    //   into O_t waits for o_free. Without that last-tile wait, split-KV
    //   prefill gave run-to-run different results.
    int o_base = 0, o_pend = 0;
    // The epilogue of a tile runs after the first P of the next tile has been
    // handed to the tensor core: the last P V of the tile then completes while
    // this warpgroup already works on the next tile (it only needs O once
    // that P V is done, and the next P V into O waits for o_free).
    // The pending tile's state lives in shared memory (16 bytes per thread:
    // m, d, query row, rows | split | keys | head), not in registers that the
    // softmax loop would have to carry.
    float4 *pend_slot = reinterpret_cast<float4 *>(smem + C::kOffPend) + threadIdx.x;
    float *pend_vs = reinterpret_cast<float *>(smem + C::kOffPendVs) + threadIdx.x;
    bool pend_on = false;
    // testing hook: a wait that runs out while the first copies and products
    // are in flight
    bool ok = p.stall_ns == 0 ||
              __all_sync(0xffffffffu, mbar_wait(&bars->never, 0, abort, &g_prefill_error, false,
                                                p.stall_ns));
    auto finish = [&]() {  // epilogue of the pending tile
      const float4 st = *pend_slot;
      const float pm = st.x, pd = st.y;
      const int qrow = __float_as_int(st.z);
      const unsigned bits = __float_as_uint(st.w);
      const int prows = static_cast<int>(bits & 0xffu);
      const int psplit = static_cast<int>((bits >> 8) & 0x7fu);
      const bool pkeys = (bits >> 15) & 1u;
      const int ph = static_cast<int>(bits >> 16);
      const size_t prow_h = static_cast<size_t>(qrow) * p.hq + ph;
      bool have_o = false;
      if (pkeys) {
        have_o = __all_sync(0xffffffffu,
                            mbar_wait(&bars->o_done[t], o_pend & 1, abort,
                                      &g_prefill_error));
        if (!have_o) {
          ok = false;
          return;
        }
      }
      const float inv = pd > 0.f ? *pend_vs / pd : 0.f;
      constexpr int kQ = D / 32;  // 32-column TMEM loads of O
      uint32_t ov[kQ][32];
      if (have_o) {
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < kQ; ++q) tmem_ld32(o_addr + 32 * q, ov[q]);
        tmem_wait_ld();
        // O_t may now be overwritten by the next tile's first P V (only tiles
        // with keys wrote O_t, and only they signal)
        tc_fence_before();
        mbar_arrive(&bars->o_free[t]);
      } else {
#pragma unroll
        for (int q = 0; q < kQ; ++q)
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[q][i] = 0u;
      }
      const float lse = pd > 0.f ? (pm + fast_log2(pd)) * kLn2 : -INFINITY;
      if (r < prows && p.num_splits > 1) {
        const size_t at = static_cast<size_t>(psplit) * p.total_q * p.hq + prow_h;
        if constexpr (kV8) {
          float *dst = p.part_o + at * D;
#pragma unroll
          for (int q = 0; q < kQ; ++q)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint32_t w[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) w[e] = __float_as_uint(__uint_as_float(ov[q][8 * i + e]) * inv);
              st_global_v8(dst + q * 32 + 8 * i, w);
            }
        } else {
          float4 *dst = reinterpret_cast<float4 *>(p.part_o + at * D);
#pragma unroll
          for (int q = 0; q < kQ; ++q)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float *o = reinterpret_cast<const float *>(&ov[q][4 * i]);
              dst[q * 8 + i] = make_float4(o[0] * inv, o[1] * inv, o[2] * inv, o[3] * inv);
            }
        }
        p.part_lse[at] = lse;
      } else if (r < prows) {
        if constexpr (kV8) {
          __nv_bfloat16 *dst = p.out + prow_h * D;
#pragma unroll
          for (int q = 0; q < kQ; ++q)
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const float *o = reinterpret_cast<const float *>(&ov[q][16 * i]);
              uint32_t w[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(o[2 * e] * inv, o[2 * e + 1] * inv);
              st_global_v8(dst + q * 32 + 16 * i, w);
            }
        } else {
          uint4 *dst = reinterpret_cast<uint4 *>(p.out + prow_h * D);
#pragma unroll
          for (int q = 0; q < kQ; ++q)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float *o = reinterpret_cast<const float *>(&ov[q][8 * i]);
              uint4 v;
              v.x = pack_bf16x2(o[0] * inv, o[1] * inv);
              v.y = pack_bf16x2(o[2] * inv, o[3] * inv);
              v.z = pack_bf16x2(o[4] * inv, o[5] * inv);
              v.w = pack_bf16x2(o[6] * inv, o[7] * inv);
              dst[q * 4 + i] = v;
            }
        }
        if (p.lse != nullptr) p.lse[prow_h] = lse;
      }
      pend_on = false;
    };
    for (int nt = 0; ok; ++nt) {
      const int slot = nt & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->tile_full[slot], (nt >> 1) & 1, abort,
                                             &g_prefill_error)))
        break;
      const Tile ti = bars->tiles[slot];
      if (!ti.valid) break;
      const int h = ti.h0 + t;
      const float c =
          p.k_scale != nullptr ? p.scale_log2 * __ldg(p.k_scale + ti.kvh) : p.scale_log2;
      const float2 c2 = make_float2(c, c);
      float m_run = t == 0 ? ti.sink_log2[0] : ti.sink_log2[1];
      float d_run = m_run != -INFINITY ? 1.f : 0.f;
      const int pos = ti.p_min + r;
      const int n = ti.n;
      for (int j = 0; j < n; ++j) {
        const int k = K + j * NT + t;  // work item: buffer k % kSBufs, its (k / kSBufs)-th use
        const int kb = k % C::kSBufs;
        const uint32_t s_addr = lane_addr + kb * kBN;
        const uint32_t p_addr = C::kSplitP ? lane_addr + C::kTmemP + kb * 64 : s_addr;
        // waits are made warp-uniform: tcgen05.ld/st below are warp-collective
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full[kb], (k / C::kSBufs) & 1,
                                               abort, &g_prefill_error))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int key0 = (ti.kt_lo + j) * kBN;
        const bool need_mask = (key0 + kBN > ti.lk) || (p.causal && key0 + kBN - 1 > ti.p_min) ||
                               (p.window > 0 && key0 <= ti.p_max - p.window);
        float s0[32], s1[32], s2[32], s3[32];
        tmem_ld32f(s_addr, s0);
        tmem_ld32f(s_addr + 32, s1);
        tmem_ld32f(s_addr + 64, s2);
        tmem_ld32f(s_addr + 96, s3);
        tmem_wait_ld();
        if (C::kSplitP) {  // the scores are in registers: the S buffer may take item k + 2's
          tc_fence_before();
          mbar_arrive(&bars->s_read[kb]);
        }
        if (need_mask) {
          // this row's visible keys form one range [lo, hi): sequence end, causal
          // bound and window; as tile columns [c_lo, c_lo + len)
          int hi = ti.lk, lo = 0;
          if (p.causal) hi = min(hi, pos + 1);
          if (p.window > 0) lo = max(lo, pos - p.window + 1);
          const int c_lo = min(max(lo - key0, 0), kBN);
          const int len = max(min(hi - key0, kBN) - c_lo, 0);
          // a 32-column chunk that every row of the warp sees whole needs no
          // test (under a causal or window bound, only the chunks that the
          // warp's rows' bounds fall in do)
          const int c_hi = c_lo + len;
          if (!__all_sync(0xffffffffu, c_lo <= 0 && c_hi >= 32)) mask32(s0, 0, c_lo, len);
          if (!__all_sync(0xffffffffu, c_lo <= 32 && c_hi >= 64)) mask32(s1, 32, c_lo, len);
          if (!__all_sync(0xffffffffu, c_lo <= 64 && c_hi >= 96)) mask32(s2, 64, c_lo, len);
          if (!__all_sync(0xffffffffu, c_lo <= 96 && c_hi >= 128)) mask32(s3, 96, c_lo, len);
        }
        const float mx = max3(fmaxf(row_max32(s0), row_max32(s1)), row_max32(s2), row_max32(s3));
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
        const float2 nb2 = make_float2(-base, -base);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
        {
          uint32_t pk[32];
          exp32(s0, c2, nb2, acc, pk, 0);
          exp32(s1, c2, nb2, acc, pk, 16);
          // separate P: P V of item k - kSBufs has finished reading this P buffer
          if (C::kSplitP && k >= C::kSBufs) {
            if (!__all_sync(0xffffffffu,
                            mbar_wait(&bars->pv_done[kb], ((k - C::kSBufs) / C::kSBufs) & 1,
                                      abort, &g_prefill_error))) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          tmem_st32(p_addr, pk);
          exp32(s2, c2, nb2, acc, pk, 0);
          exp32(s3, c2, nb2, acc, pk, 16);
          tmem_st32(p_addr + 32, pk);
        }
        const float2 a01 = __fadd2_rn(acc[0], acc[1]), a23 = __fadd2_rn(acc[2], acc[3]);
        const float2 a03 = __fadd2_rn(a01, a23);
        d_run += a03.x + a03.y;
        tmem_wait_st();
        // O_t holds P_0..P_{j-1} V; it must be complete before it is rescaled
        if (j > 0 && (j == n - 1 || __any_sync(0xffffffffu, rescale))) {
          if (!__all_sync(0xffffffffu, mbar_wait(&bars->o_done[t], (o_base + j - 1) & 1, abort,
                                                 &g_prefill_error))) {
            ok = false;
            break;
          }
          // one lane's rescale makes the whole warp run the (collective) O round
          // trip; lanes that did not move their maximum multiply by alpha = 1
          if (__any_sync(0xffffffffu, rescale)) {
            tc_fence_after();
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
              uint32_t ov[32];
              tmem_ld32(o_addr + q * 32, ov);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
              tmem_st32(o_addr + q * 32, ov);
            }
            tmem_wait_st();
          }
        }
        tc_fence_before();
        mbar_arrive(&bars->p_full[kb]);
        if (j == 0 && pend_on) {  // the previous tile's epilogue, behind this P
          finish();
          if (!ok) break;
        }
      }
      if (!ok) break;
      if (pend_on) {  // a tile without keys: nothing to hide the epilogue behind
        finish();
        if (!ok) break;
      }
      pend_on = true;
      *pend_slot = make_float4(
          m_run, d_run, __int_as_float(ti.q0 + ti.qt * kBM + r),
          __uint_as_float(static_cast<unsigned>(ti.rows) | (static_cast<unsigned>(ti.split) << 8) |
                          (n > 0 ? 1u << 15 : 0u) | (static_cast<unsigned>(h) << 16)));
      *pend_vs = p.v_scale != nullptr ? __ldg(p.v_scale + ti.kvh) : 1.f;
      mbar_arrive(&bars->tile_empty[slot]);
      if (n > 0) {
        o_pend = o_base + n - 1;
        o_base += n;
      }
      K += NT * n;
    }
    if (ok && pend_on) finish();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// bf16 V -> fp16 copy for the P V product (8 elements per thread per step).
// The prefill kernel launched after it may start at once (programmatic
// dependent launch): only its V producer waits for this grid.
__global__ void __launch_bounds__(256) convert_v_kernel(const uint4 *__restrict__ src,
                                                        uint4 *__restrict__ dst, int64_t n8) {
  asm volatile("griddepcontrol.launch_dependents;");
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    dst[i] = bf16x8_to_f16x8(src[i]);
}

}  // namespace

// ---------------------------------------------------------------- host side

cudaError_t launch_tile_list(const int32_t *cu, int batch, int max_tiles, unsigned *pairs,
                             int *num_pairs, unsigned *counter, cudaStream_t stream) {
  build_worklist_kernel<<<1, 1024, 0, stream>>>(cu, batch, max_tiles, pairs, num_pairs, counter);
  return cudaGetLastError();
}

namespace {

// testing hook (sinkattn_debug_stall_waits): stall_ns of later launches
std::atomic<uint64_t> g_stall_ns{0};

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Workspace pieces (head dimension d). Every piece starts on a 256-byte boundary.
size_t vcopy_bytes(int64_t total_k, int hkv, int d) {  // fp16 copy of V
  return round256(static_cast<size_t>(total_k) * hkv * d * 2);
}
size_t schedule_bytes(int batch, int64_t total_q) {  // tile counter + work list
  return 256 + round256(static_cast<size_t>(total_q / kBM + batch) * 4);
}
size_t partial_o_bytes(int64_t total_q, int hq, int splits, int d) {
  return splits > 1 ? round256(static_cast<size_t>(splits) * total_q * hq * d * 4) : 0;
}
size_t partials_bytes(int64_t total_q, int hq, int splits, int d) {  // o, then lse
  return splits > 1 ? partial_o_bytes(total_q, hq, splits, d) +
                          round256(static_cast<size_t>(splits) * total_q * hq * 4)
                    : 0;
}
// Paged staging: K (bf16) or V (fp16) of up to batch * max_seqlen_k rows plus
// a zeroed 128-row tail.
int64_t paged_stage_rows(int batch, int max_seqlen_k) {
  return static_cast<int64_t>(batch) * max_seqlen_k + kBM;
}
size_t paged_stage_bytes(int batch, int max_seqlen_k, int hkv, int d) {
  return round256(static_cast<size_t>(paged_stage_rows(batch, max_seqlen_k)) * hkv * d * 2);
}

}  // namespace

int prefill_plan_splits(int requested, int batch, int64_t total_q, int max_seqlen_q,
                        int max_seqlen_k, int hq, int hkv, int window, int head_dim) {
  if (requested > 0) return requested < kMaxPrefillSplits ? requested : kMaxPrefillSplits;
  const int nt = head_dim == 64 && (hq / hkv) % 2 == 0 ? 2 : 1;
  const int64_t qtiles = (max_seqlen_q + kBM - 1) / kBM;
  const int64_t pairs = std::min<int64_t>(total_q / kBM + batch, batch * qtiles);
  const int64_t items = pairs * (hq / nt);
  int64_t kv_tiles = (max_seqlen_k + kBN - 1) / kBN;
  if (window > 0)
    kv_tiles = std::min<int64_t>(kv_tiles, (static_cast<int64_t>(window) + kBM - 1) / kBN + 2);
  const int64_t sms = sm_count();
  // Enough items already, or too few keys to be worth cutting.
  if (items <= 0 || items >= 2 * sms || kv_tiles < 32) return 1;
  // Cost model: the items run in waves over the SMs; an item costs its share
  // of key tiles plus about 4 tiles of fixed work (Q load, pipeline fill and
  // drain, epilogue). The merge pass is small next to that.
  int best = 1;
  int64_t best_cost = INT64_MAX;
  const int64_t max_s = std::min<int64_t>(kMaxPrefillSplits, kv_tiles / 16);
  for (int64_t s = 1; s <= max_s; ++s) {
    const int64_t waves = (items * s + sms - 1) / sms;
    const int64_t cost = waves * ((kv_tiles + s - 1) / s + 4);
    if (cost < best_cost) {
      best_cost = cost;
      best = static_cast<int>(s);
    }
  }
  return best;
}

size_t prefill_workspace_bytes(int batch, int64_t total_q, int64_t total_k, int hq, int hkv,
                               int splits, int head_dim) {
  return vcopy_bytes(total_k, hkv, head_dim) + schedule_bytes(batch, total_q) +
         partials_bytes(total_q, hq, splits, head_dim);
}

// Paged prefill workspace: K staging, V staging, the sequence offsets, the
// schedule, the split partials.
size_t prefill_paged_workspace_bytes(int batch, int64_t total_q, int max_seqlen_k, int hq,
                                     int hkv, int splits, int head_dim) {
  return 2 * paged_stage_bytes(batch, max_seqlen_k, hkv, head_dim) +
         round256(static_cast<size_t>(batch + 1) * 4) + schedule_bytes(batch, total_q) +
         partials_bytes(total_q, hq, splits, head_dim);
}

namespace {

// cu_k[b] = sum of min(seqlens_k[i], max_seqlen_k) over i < b (one block).
__global__ void __launch_bounds__(1024) seqlen_offsets_kernel(const int32_t *seqlens_k, int batch,
                                                               int max_seqlen_k, int32_t *cu_k) {
  int carry = 0;
  for (int base = 0; base < batch; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int len = 0;
    if (b < batch) {
      len = seqlens_k[b];
      if (len < 0 || len > max_seqlen_k) {
        atomicExch(&g_prefill_error, kErrBadLength);
        len = min(max(len, 0), max_seqlen_k);
      }
    }
    int total = 0;
    const int ex = block_exclusive_scan(len, &total);
    if (b < batch) cu_k[b] = carry + ex;
    carry += total;
    __syncthreads();  // warp_sums is reused by the next chunk
  }
  if (threadIdx.x == 0) cu_k[batch] = carry;
}

// e4m3 -> bf16 for 8 elements (exact: 3 mantissa bits, exponents well
// inside bf16's range)
__device__ __forceinline__ uint4 e4m3x8_to_bf16x8(uint2 x) {
  uint32_t h[4];
  e4m3x4_to_f16x4(x.x, h[0], h[1]);
  e4m3x4_to_f16x4(x.y, h[2], h[3]);
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h[i]));
    o[i] = pack_bf16x2(f.x, f.y);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// e4m3 -> fp16 for 8 elements (exact)
__device__ __forceinline__ uint4 e4m3x8_to_f16x8(uint2 x) {
  uint4 r;
  e4m3x4_to_f16x4(x.x, r.x, r.y);
  e4m3x4_to_f16x4(x.y, r.z, r.w);
  return r;
}

// Paged K/V -> contiguous staging, one warp per token (all KV heads): K as
// bf16, V converted to fp16 (clamped to +-65504) for the P V product. With
// kFp8 the cache holds e4m3 codes, staged as their exact values (the scales
// are applied by the attention kernel). Rows [total, total + 128) are zeroed
// so that a tile running past the last sequence reads zeros.
template <bool kFp8>
__global__ void __launch_bounds__(256) gather_paged_kernel(
    const void *__restrict__ kc, const void *__restrict__ vc,
    const int32_t *__restrict__ block_table, const int32_t *__restrict__ cu_k, int batch,
    int max_pages, int page_size, int num_pages, int hkv, int d, int64_t cap_rows,
    __nv_bfloat16 *__restrict__ k_out,
    __half *__restrict__ v_out) {
  const int lane = threadIdx.x & 31;
  const int64_t total = cu_k[batch];
  const int64_t end = total + kBM < cap_rows ? total + kBM : cap_rows;
  const int chunks = hkv * (d / 8);  // 16-byte chunks per token row of all heads
  for (int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32; r < end;
       r += static_cast<int64_t>(gridDim.x) * blockDim.x / 32) {
    uint4 *kd = reinterpret_cast<uint4 *>(k_out + r * hkv * d);
    uint4 *vd = reinterpret_cast<uint4 *>(v_out + r * hkv * d);
    int page = -1, slot = 0;
    if (r < total) {
      int lo = 0, hi = batch;  // sequence b with cu_k[b] <= r < cu_k[b + 1]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cu_k[mid] <= r) lo = mid; else hi = mid;
      }
      const int j = static_cast<int>(r - cu_k[lo]);
      page = block_table[static_cast<size_t>(lo) * max_pages + j / page_size];
      slot = j % page_size;
      if (page < 0 || page >= num_pages) {
        if (lane == 0) atomicExch(&g_prefill_error, kErrBadPage);
        page = -1;
      }
    }
    if (page < 0) {
      for (int c = lane; c < chunks; c += 32) {
        kd[c] = make_uint4(0u, 0u, 0u, 0u);
        vd[c] = make_uint4(0u, 0u, 0u, 0u);
      }
      continue;
    }
    for (int c = lane; c < chunks; c += 32) {
      const int h = c / (d / 8), e = c % (d / 8);
      const size_t src = ((static_cast<size_t>(page) * hkv + h) * page_size + slot) * d;
      if constexpr (kFp8) {
        kd[c] = e4m3x8_to_bf16x8(reinterpret_cast<const uint2 *>(
            static_cast<const uint8_t *>(kc) + src)[e]);
        vd[c] = e4m3x8_to_f16x8(reinterpret_cast<const uint2 *>(
            static_cast<const uint8_t *>(vc) + src)[e]);
      } else {
        kd[c] = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(kc) + src)[e];
        vd[c] = bf16x8_to_f16x8(
            reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(vc) + src)[e]);
      }
    }
  }
}

// Everything after the K/V staging: tensor maps, the work list, the kernel
// and, with splits, the merge. k (bf16) and v16 (fp16) are [k_rows, hkv, 64];
// cu_k may live on the device only; sched is the schedule area (tile counter +
// work list), followed by the split partials.
// v_src / n8: bf16 V to convert into v16 (n8 16-byte chunks) after the work
// list is built, overlapped with the start of the prefill kernel; n8 = 0:
// v16 is ready.
cudaError_t launch_core(const PrefillLaunch &a, const void *k, const void *v16, int64_t k_rows,
                        const int32_t *cu_k, uint8_t *sched, cudaStream_t stream,
                        bool *encode_failed, const void *v_src = nullptr, int64_t n8 = 0) {
  const int max_qtiles = (a.max_seqlen_q + kBM - 1) / kBM;
  EncodeTiledFn fn = get_encode_fn();
  CUtensorMap tq, tk, tv;
  const CUtensorMapDataType bf16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  // With no keys at all nothing reads K or V; the maps then point at q.
  const void *kbase = k_rows > 0 ? k : a.q;
  const void *vbase = k_rows > 0 ? v16 : a.q;
  const int d = a.head_dim;
  if (fn == nullptr || !encode_rows_heads(fn, &tq, a.q, a.total_q, a.hq, bf16, d) ||
      !encode_rows_heads(fn, &tk, kbase, k_rows, a.hkv, bf16, d) ||
      !encode_rows_heads(fn, &tv, vbase, k_rows, a.hkv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, d)) {
    *encode_failed = true;
    return cudaErrorInvalidValue;
  }
  Params p;
  p.cu_q = a.cu_q;
  p.cu_k = cu_k;
  p.batch = a.batch;
  p.hq = a.hq;
  p.group = a.hq / a.hkv;
  p.causal = a.causal ? 1 : 0;
  p.window = a.window;
  p.max_qtiles = max_qtiles;
  p.sinks = a.sinks;
  p.scale_log2 = a.scale * kLog2e;
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.lse = a.lse;
  p.work_counter = reinterpret_cast<unsigned int *>(sched);
  int *num_pairs = reinterpret_cast<int *>(sched + 4);
  unsigned *pairs = reinterpret_cast<unsigned *>(sched + 256);
  p.work_pairs = pairs;
  p.num_pairs = num_pairs;
  const int splits = a.num_splits > 1 ? a.num_splits : 1;
  p.num_splits = splits;
  p.total_q = static_cast<int>(a.total_q);
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.stall_ns = g_stall_ns.load();
  uint8_t *part = sched + schedule_bytes(a.batch, a.total_q);
  p.part_o = splits > 1 ? reinterpret_cast<float *>(part) : nullptr;
  p.part_lse = splits > 1 ? reinterpret_cast<float *>(
                                part + partial_o_bytes(a.total_q, a.hq, splits, d))
                          : nullptr;
  const bool v8 = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0 &&
                  (reinterpret_cast<uintptr_t>(p.part_o) & 31u) == 0;
  // head_dim 64: two heads per item when the group size is even; 128: one
  const int nt = d == 64 && p.group % 2 == 0 ? 2 : 1;
  build_worklist_kernel<<<1, 1024, 0, stream>>>(a.cu_q, a.batch, max_qtiles, pairs, num_pairs,
                                                p.work_counter);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const bool pdl = n8 > 0;
  if (pdl) {
    const int64_t blocks = (n8 + 255) / 256;
    convert_v_kernel<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(
        static_cast<const uint4 *>(v_src), static_cast<uint4 *>(const_cast<void *>(v16)), n8);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // upper bound on the number of work items, for the grid size
  const int64_t max_pairs = a.total_q / kBM + a.batch;
  const int64_t max_work = max_pairs * (a.hq / nt) * splits;
  // one resident CTA per SM, two for the dual (one head, head_dim 64) kernel
  const int num_ctas = sm_count() * (nt == 1 && d == 64 ? 2 : 1);
  const unsigned grid = static_cast<unsigned>(max_work < num_ctas ? max_work : num_ctas);
  // launch one of the kernels, overlapping the V conversion when there is one
  auto go = [&](auto kernel, int threads, int smem_bytes) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, p);
  };
  // setmaxnreg.inc waits until the registers exist: a kernel with a register
  // split must be launched with at least the split's total, or its softmax
  // warps would never start.
  auto launch = [&](auto ntc, auto dc, auto v8c) -> cudaError_t {
    constexpr int NT = decltype(ntc)::value, D = decltype(dc)::value;
    constexpr bool V8 = decltype(v8c)::value;
    using CC = Cfg<NT, D>;
    auto kernel = prefill_kernel<NT, D, V8>;
    cudaError_t e2 =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, CC::kSmemBytes);
    if (e2 != cudaSuccess) return e2;
    constexpr int need = NT == 2 ? kRegsOther2 * 128 + kRegsSoftmax2 * 256
                         : D == 64 ? kRegsOtherD * 128 + kRegsSoftmaxD * 128
                                   : 0;
    if (need > 0) {
      static int launch_regs = -1;  // one per instantiation
      if (launch_regs < 0) {
        cudaFuncAttributes attr;
        e2 = cudaFuncGetAttributes(&attr, kernel);
        if (e2 != cudaSuccess) return e2;
        launch_regs = attr.numRegs;
      }
      if (launch_regs * CC::kThreads < need) return cudaErrorNotSupported;
    }
    return go(kernel, CC::kThreads, CC::kSmemBytes);
  };
  auto launch_v8 = [&](auto ntc, auto dc) {
    return v8 ? launch(ntc, dc, std::true_type()) : launch(ntc, dc, std::false_type());
  };
  if (nt == 2)
    e = launch_v8(std::integral_constant<int, 2>(), std::integral_constant<int, 64>());
  else if (d == 64)
    e = launch_v8(std::integral_constant<int, 1>(), std::integral_constant<int, 64>());
  else
    e = launch_v8(std::integral_constant<int, 1>(), std::integral_constant<int, 128>());
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess || splits == 1) return e;
  // split 0 carried the sink: the merge adds no sink of its own
  return launch_merge(p.part_o, p.part_lse, splits, a.total_q, a.hq, d, nullptr, a.out, a.lse,
                      stream);
}

}  // namespace

cudaError_t launch_prefill(const PrefillLaunch &a, cudaStream_t stream, bool *encode_failed) {
  *encode_failed = false;
  const int max_qtiles = (a.max_seqlen_q + kBM - 1) / kBM;
  if (a.batch == 0 || a.total_q == 0 || max_qtiles == 0) return cudaSuccess;
  // the bf16 -> fp16 copy of V runs after the work list, overlapped with the
  // prefill kernel's start
  const int64_t n8 = a.total_k * a.hkv * a.head_dim / 8;
  uint8_t *ws = static_cast<uint8_t *>(a.v_f16);
  return launch_core(a, a.k, a.v_f16, a.total_k, a.cu_k,
                     ws + vcopy_bytes(a.total_k, a.hkv, a.head_dim), stream, encode_failed, a.v,
                     n8);
}

cudaError_t launch_prefill_paged(const PrefillPagedLaunch &a, cudaStream_t stream,
                                 bool *encode_failed) {
  *encode_failed = false;
  const PrefillLaunch &c = a.base;
  const int max_qtiles = (c.max_seqlen_q + kBM - 1) / kBM;
  if (c.batch == 0 || c.total_q == 0 || max_qtiles == 0) return cudaSuccess;
  uint8_t *ws = static_cast<uint8_t *>(a.workspace);
  const size_t stage = paged_stage_bytes(c.batch, c.max_seqlen_k, c.hkv, c.head_dim);
  __nv_bfloat16 *k_st = reinterpret_cast<__nv_bfloat16 *>(ws);
  __half *v_st = reinterpret_cast<__half *>(ws + stage);
  int32_t *cu_k = reinterpret_cast<int32_t *>(ws + 2 * stage);
  uint8_t *sched = ws + 2 * stage + round256(static_cast<size_t>(c.batch + 1) * 4);
  seqlen_offsets_kernel<<<1, 1024, 0, stream>>>(a.seqlens_k, c.batch, c.max_seqlen_k, cu_k);
  const int64_t cap = paged_stage_rows(c.batch, c.max_seqlen_k);
  const int64_t warps = cap < sm_count() * 64 ? cap : sm_count() * 64;
  const unsigned blocks = static_cast<unsigned>((warps + 7) / 8);
  if (a.fp8)
    gather_paged_kernel<true><<<blocks, 256, 0, stream>>>(
        a.k_cache, a.v_cache, a.block_table, cu_k, c.batch, a.max_pages, a.page_size, a.num_pages,
        c.hkv, c.head_dim, cap, k_st, v_st);
  else
    gather_paged_kernel<false><<<blocks, 256, 0, stream>>>(
        a.k_cache, a.v_cache, a.block_table, cu_k, c.batch, a.max_pages, a.page_size, a.num_pages,
        c.hkv, c.head_dim, cap, k_st, v_st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_core(c, k_st, v_st, cap, cu_k, sched, stream, encode_failed);
}

cudaError_t prefill_set_stall(uint64_t ns) {
  g_stall_ns.store(ns);
  return cudaSuccess;
}

cudaError_t prefill_read_error(cudaStream_t stream, int *code) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(code, g_prefill_error, sizeof(int));
  const int zero = 0;
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof(int));
  return e;
}

}  // namespace sinkattn
