// Split-KV decode for sink attention: one query token per sequence over a
// contiguous or paged KV cache in bf16, or in fp8 e4m3 with per-KV-head
// scales.
//
// Page "GPT-OSS on day 0", section "Kernels for GPT-OSS / Sink Attention":
// the online softmax keeps a running maximum m and a running denominator d;
// the head's sink is folded in by starting m at the sink (with d = 1) instead
// of at -inf, and when the KV sequence is cut into blocks only one block may
// start that way. Page "CuTeDSL at Perplexity", section "Prefill and decode
// specialisation": decode is bound by the DRAM traffic of the KV cache, so it
// gets its own kernel and grid.
//
// Block = (split s, KV head g, sequence b), 4 warps. The block owns a chunk of
// the visible keys; each warp streams 32-token slabs of K and V (slabs w,
// w+4, ...) into its own shared-memory ring (two or three stages, per cache
// form) with 16-byte cp.async copies, so no block-wide barrier sits in the
// loop. All group query heads of
// KV head g (up to 8) are served from one read of each K/V byte:
//
//   S^T[16 tokens x 8 heads] = K[16 x 64] . Q^T   (mma.sync m16n8k16, N = heads)
//   O^T[64 dims x 8 heads]  += V^T . P^T          (P^T re-used as the B operand
//                                                  after an in-register 8x8
//                                                  transpose, movmatrix)
//
// fp8 cache (page "GPT-OSS on day 0": FP8 serving): the ring holds e4m3 slabs
// (half the bytes, 64-byte rows) and the MMA fragments are built straight
// from them in registers (e4m3 -> fp16 is exact); the MMAs run in fp16 (q
// converted once, P as one fp16 term). Two relabelings make every fragment a
// plain load: the 64 dims of q and K are visited in the order that puts a
// thread's four K bytes of one k-step side by side (a dot product does not
// care about the order), and V^T's MMA rows stand for dims 2r and 2r+1 of each
// 16-dim tile (undone when O is stored). The K scale folds into the softmax
// scale, the V scale into the final normalisation.
//
// The per-warp states (m, d, O) are combined in shared memory; a sequence with
// one block writes the final bf16 output directly, otherwise each block writes
// a normalised fp32 partial and its log-sum-exp, and the last block to arrive
// (per-(sequence, KV head) counter, no grid barrier) merges them
// (page "CuTeDSL at Perplexity", section "Grid synchronization": prefer kernel
// boundaries or local counters over grid-wide barriers).
#include <math.h>

#include <mutex>
#include <type_traits>

#include "../../include/sinkattn.h"
#include "launch.h"
#include "ptx.cuh"

namespace sinkattn {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxGroup = 8;
// Longest visible span (tokens) decoded one warp per (sequence, KV head).
// Measured on GB300 at a 128-token window: 25.2 vs 30.3 us on the paged
// decode workload, 10.9 vs 12.9 us on the contiguous one; at 256 and 512
// tokens the four-warp blocks are as fast or faster.
constexpr int kPairMaxSpan = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Shapes for head dimension D (64 or 128). A warp step covers kSlab tokens:
// 32 at D = 64, 16 at D = 128, so that a slab of K and V is the same number
// of bytes for both: 8 KB per stage for bf16, 4 KB for fp8 (ring depths
// and blocks per SM in Ring below). kHalfSlab: 16-token steps at D = 64 too
// (the one-warp-per-pair bf16 form, whose rings must be small).
template <int D, bool kHalfSlab = false>
struct DCfg {
  static constexpr int kSlab = D == 64 && !kHalfSlab ? 32 : 16;
  static constexpr int kMT = kSlab / 16;         // 16-token m-tiles per slab
  static constexpr int kKS = D / 16;             // k-steps of Q K^T, dim tiles of P V
  static constexpr int kRowBytes = D * 2;        // bf16 row
  static constexpr int kSlabBytes = kSlab * kRowBytes;
  static constexpr int kStageBytes = 2 * kSlabBytes;
  static constexpr int kRowBytes8 = D;           // fp8 row
  static constexpr int kSlabBytes8 = kSlab * kRowBytes8;
  static constexpr int kStageBytes8 = 2 * kSlabBytes8;
  static constexpr int kOutPer = D / 16;         // output dims per thread in the epilogue
};

// Per-warp ring depth and resident blocks per SM for each cache form,
// measured on GB300 (same results bitwise, only the schedule differs):
// - contiguous bf16: three stages at two blocks per SM (101.4 us on the
//   contiguous decode workload; 104.9 us with two stages at three blocks);
// - paged bf16 (2 KB pieces per 16-token page): two stages at three blocks
//   (1218 us vs 1280 us on the paged decode workload, 2% at head_dim 128);
// - contiguous fp8 at head_dim 64: two stages at five blocks (64 us vs
//   65 us); paged fp8 keeps three stages at four blocks (639 us vs 651 us
//   with five), as does head_dim 128 over fp8;
// - one warp per pair, bf16 at head_dim 64: three stages of 16 tokens (4 KB)
//   at four blocks per SM. The paged window-128 workload (2048 pairs, 512
//   blocks) then runs in one wave of 608 block slots instead of two of 456
//   with 32-token slabs at three blocks.
template <int D, bool kPaged, bool kFp8, bool kPair = false>
struct Ring {
  static constexpr bool kHalfSlab = kPair && !kFp8 && D == 64;
  using C = DCfg<D, kHalfSlab>;
  static constexpr bool kFp8Wide = kFp8 && !kPaged && D == 64;
  static constexpr int kStages =
      kHalfSlab ? 3 : kFp8 ? (kFp8Wide ? 2 : 3) : (kPaged ? 2 : 3);
  static constexpr int kBlocks =
      kHalfSlab ? 4 : kFp8 ? (kFp8Wide ? 5 : 4) : (kPaged ? 3 : 2);
  static constexpr int kSmemBytes = kWarps * kStages * (kFp8 ? C::kStageBytes8 : C::kStageBytes);
  // the warps' states are combined in the ring's memory after the loop (in
  // the one-warp-per-pair form each warp uses its own quarter)
  static_assert(kSmemBytes >= (2 + D) * kWarps * kMaxGroup * 4, "combine area");
};

struct Params {
  const __nv_bfloat16 *q, *k, *v;
  const uint8_t *k8, *v8;            // fp8 cache
  const float *k_scale, *v_scale;    // fp8: per KV head, or null
  const int32_t *kv_indptr, *block_table, *seqlens_k;
  int max_pages, page_size;
  int page_shift;  // log2(page_size) when it is a power of two, else -1
  int batch, hq, hkv, group, window, chunk;
  int nht;  // tiles of up to 8 query heads per KV head
  const float *sinks;
  float scale_log2;
  __nv_bfloat16 *out;
  float *lse;
  float *part_o, *part_lse;
  unsigned int *counters;
};

// Page ids of one block's token range are staged in shared memory once per
// block (one coalesced read of the block table) so the per-row address needs
// no dependent global load; ranges longer than this read the table directly.
constexpr int kMaxBlockPages = 1024;

__device__ __forceinline__ int page_index(const Params &p, int j) {
  return p.page_shift >= 0 ? j >> p.page_shift : j / p.page_size;
}
__device__ __forceinline__ int page_slot(const Params &p, int j) {
  return p.page_shift >= 0 ? j & (p.page_size - 1) : j % p.page_size;
}

// Element offset of row (token j, KV head g) of sequence b in the K/V cache.
// Paged: pages[] holds the ids of pages pg0.. when `staged`.
template <int D, bool kPaged>
__device__ __forceinline__ size_t kv_row(const Params &p, int b, int kv_base, int j, int g,
                                         const int *pages, int pg0, bool staged) {
  if (kPaged) {
    const int pi = page_index(p, j);
    const int page = staged ? pages[pi - pg0]
                            : __ldg(p.block_table + static_cast<size_t>(b) * p.max_pages + pi);
    return ((static_cast<size_t>(page) * p.hkv + g) * p.page_size + page_slot(p, j)) * D;
  }
  return (static_cast<size_t>(kv_base + j) * p.hkv + g) * D;
}

// bf16 rows (128 or 256 bytes): 16-byte chunks XOR-swizzled by row so that
// ldmatrix of 8 rows of one chunk column touches 8 different bank groups.
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * DCfg<D>::kRowBytes + ((chunk ^ (row & 7)) << 4));
}

// fp8 rows (64 or 128 bytes): chunks XOR-swizzled by row / 2 (four chunks) or
// by row (eight chunks), which makes the fragment loads below free of bank
// conflicts.
template <int D>
__device__ __forceinline__ int swz8(int row, int chunk) {
  const int x = D == 64 ? ((row >> 1) & 3) : (row & 7);
  return row * DCfg<D>::kRowBytes8 + ((chunk ^ x) << 4);
}

// Zeroes the split-merge counters of one decode call. It allows the decode
// grid that follows to launch immediately (griddepcontrol.launch_dependents);
// the decode waits for this grid (griddepcontrol.wait) before its first
// counter access.
__global__ void __launch_bounds__(256) zero_counters_kernel(unsigned int *c, int64_t n) {
  asm volatile("griddepcontrol.launch_dependents;");
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    c[i] = 0u;
}

// kPair: short spans (a sliding window, short contexts). Each warp owns one
// (sequence, KV head) and streams its whole visible span through its own
// ring, so a block serves four pairs and no barrier spans the block; with
// four warps per pair a 128-token window gives each warp a single slab, and
// the many short blocks run in latency-bound waves.
template <int D, bool kPaged, bool kFp8, bool kPair>
__global__ void __launch_bounds__(kThreads, (Ring<D, kPaged, kFp8, kPair>::kBlocks))
    decode_kernel(const Params p) {
  using R = Ring<D, kPaged, kFp8, kPair>;
  using C = typename R::C;
  constexpr int kStages = R::kStages;
  constexpr int kSlab = C::kSlab, kMT = C::kMT, kKS = C::kKS;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lr = lane >> 2, lc = lane & 3;  // mma fragment row / column group
  int split = 0, g, b, ht;
  if (kPair) {
    const int pair = static_cast<int>(blockIdx.x) * kWarps + warp;
    if (pair >= p.batch * p.hkv * p.nht) return;  // no pair for this warp (no block barrier follows)
    b = pair / (p.hkv * p.nht);
    const int gh = pair - b * p.hkv * p.nht;
    g = gh / p.nht;
    ht = gh - g * p.nht;
  } else {
    split = blockIdx.x;
    g = static_cast<int>(blockIdx.y) / p.nht;
    ht = static_cast<int>(blockIdx.y) - g * p.nht;
    b = blockIdx.z;
  }
  // this block's query heads: gt (at most 8) heads from hbase, tile ht of
  // KV head g's group
  const int hbase = g * p.group + ht * kMaxGroup;
  const int gt = min(kMaxGroup, p.group - ht * kMaxGroup);
  const int cidx = (b * p.hkv + g) * p.nht + ht;  // split-merge counter

  int kv_base = 0, L;
  if (kPaged) {
    L = p.seqlens_k[b];
  } else {
    kv_base = p.kv_indptr[b];
    L = p.kv_indptr[b + 1] - kv_base;
  }
  const int lo = p.window > 0 ? max(0, L - p.window) : 0;
  const int nkv = max(0, L - lo);
  // A context longer than the host's max_seqlen_k bound would need more
  // blocks than the grid has: such a sequence gets longer blocks instead.
  int chunk = kPair ? max(nkv, 1) : p.chunk;
  if (!kPair && (nkv + chunk - 1) / chunk > static_cast<int>(gridDim.x)) {
    const int unit = kWarps * kSlab;
    chunk = ((nkv + gridDim.x - 1) / gridDim.x + unit - 1) / unit * unit;
  }
  const int nsplit = max(1, (nkv + chunk - 1) / chunk);
  if (split >= nsplit) return;
  const int t0 = lo + split * chunk;
  const int t1 = min(L, t0 + chunk);
  const int nslab = (max(0, t1 - t0) + kSlab - 1) / kSlab;

  __shared__ int s_pages[kPaged && !kPair ? kMaxBlockPages : 1];
  int pg0 = 0;
  bool staged = false;
  if (kPaged && !kPair) {
    pg0 = page_index(p, t0);
    const int npg = t1 > t0 ? page_index(p, t1 - 1) - pg0 + 1 : 0;
    staged = npg <= kMaxBlockPages;
    if (staged)
      for (int i = threadIdx.x; i < npg; i += kThreads)
        s_pages[i] = p.block_table[static_cast<size_t>(b) * p.max_pages + pg0 + i];
    __syncthreads();
  }
  // slabs of this warp: w, w + 4, ... of the block's range (one pair per
  // warp: all of them)
  const int slab_first = kPair ? 0 : warp, slab_step = kPair ? 1 : kWarps;
  const int my_slabs =
      kPair ? nslab : (warp < nslab ? (nslab - warp + kWarps - 1) / kWarps : 0);

  // Q^T as the B operand of S^T = K Q^T: lane (lr, lc) holds head lr,
  // dims ks*16 + 2lc + {0,1} and + 8 (fp8 cache: as fp16, clamped to its range).
  uint32_t qf[kKS][2];
  {
    const bool valid = lr < gt;
    const __nv_bfloat16 *qrow = p.q + (static_cast<size_t>(b) * p.hq + hbase + (valid ? lr : 0)) * D;
    auto frag = [&](int at) -> uint32_t {
      if (!valid) return 0u;
      const uint32_t x = *reinterpret_cast<const uint32_t *>(qrow + at);
      if (!kFp8) return x;
      const float lim = 65504.f;
      return pack_f16x2(fminf(fmaxf(bf16_lo(x), -lim), lim), fminf(fmaxf(bf16_hi(x), -lim), lim));
    };
#pragma unroll
    for (int ks = 0; ks < kKS; ++ks) {
      // fp8: k positions 2lc, 2lc+1 / 2lc+8, 2lc+9 of k-step ks stand for
      // dims f, f+1 / f+2, f+3 with f = 16 (lc + 4 (ks / 4)) + 4 (ks % 4), so
      // that one 16-byte load of K row r at chunk lc + 4 (ks / 4) holds the
      // row's A-fragment bytes of four k-steps (the K fragments use the same
      // order; a dot product does not depend on it)
      const int f = kFp8 ? 16 * (lc + 4 * (ks >> 2)) + 4 * (ks & 3) : ks * 16 + 2 * lc;
      qf[ks][0] = frag(f);
      qf[ks][1] = frag(kFp8 ? f + 2 : f + 8);
    }
  }
  // fp8: the K scale multiplies every score, the V scale every output
  const float score_log2 = kFp8 && p.k_scale != nullptr ? p.scale_log2 * p.k_scale[g]
                                                         : p.scale_log2;
  const float out_scale = kFp8 && p.v_scale != nullptr ? p.v_scale[g] : 1.f;

  // Online-softmax state for heads 2lc and 2lc+1 (log2 domain). The sink
  // initialises block 0, warp 0: m = sink, d = 1 (d kept by lane row 0 only,
  // since d is summed over the 8 lane rows at the end).
  float m0 = -INFINITY, m1 = -INFINITY, d0 = 0.f, d1 = 0.f;
  if (p.sinks != nullptr && split == 0 && (kPair || warp == 0)) {
    const int h0 = min(2 * lc, gt - 1), h1 = min(2 * lc + 1, gt - 1);
    m0 = p.sinks[hbase + h0] * kLog2e;
    m1 = p.sinks[hbase + h1] * kLog2e;
    if (lr == 0) d0 = d1 = 1.f;
  }
  float o[kKS][4];
#pragma unroll
  for (int i = 0; i < kKS; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[i][e] = 0.f;

  const uint32_t wbase =
      smem_u32(smem) + warp * kStages * (kFp8 ? C::kStageBytes8 : C::kStageBytes);

  auto load_slab = [&](int i) {
    const int slab0 = t0 + (slab_first + i * slab_step) * kSlab;
    if (kFp8) {
      // kSlab rows of D/16 chunks: 128 chunks, four per lane
      constexpr int kCols = D / 16;
      const uint32_t kdst = wbase + (i % kStages) * C::kStageBytes8;
      const uint32_t vdst = kdst + C::kSlabBytes8;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int idx = r * 32 + lane;
        const int row = idx / kCols, col = idx % kCols;
        const int j = slab0 + row;
        const bool ok = j < t1;
        const size_t off =
            ok ? kv_row<D, kPaged>(p, b, kv_base, j, g, s_pages, pg0, staged) + col * 16 : 0;
        cp_async_16(kdst + swz8<D>(row, col), p.k8 + off, ok ? 16u : 0u);
        cp_async_16(vdst + swz8<D>(row, col), p.v8 + off, ok ? 16u : 0u);
      }
      return;
    }
    // kSlab rows of D/8 chunks: 256 chunks, eight per lane (128, four per
    // lane, in 16-token slabs at D = 64)
    constexpr int kCols = D / 8;
    const uint32_t kdst = wbase + (i % kStages) * C::kStageBytes;
    const uint32_t vdst = kdst + C::kSlabBytes;
#pragma unroll
    for (int r = 0; r < kSlab * kCols / 32; ++r) {
      const int idx = r * 32 + lane;
      const int row = idx / kCols, col = idx % kCols;
      const int j = slab0 + row;
      const bool ok = j < t1;
      const size_t off =
          ok ? kv_row<D, kPaged>(p, b, kv_base, j, g, s_pages, pg0, staged) + col * 8 : 0;
      cp_async_16(kdst + swz<D>(row, col), p.k + off, ok ? 16u : 0u);
      cp_async_16(vdst + swz<D>(row, col), p.v + off, ok ? 16u : 0u);
    }
  };

#pragma unroll
  for (int i = 0; i < kStages - 1; ++i) {
    if (i < my_slabs) load_slab(i);
    cp_async_commit();
  }

  for (int it = 0; it < my_slabs; ++it) {
    cp_async_wait<kStages - 2>();
    __syncwarp();
    if (it + kStages - 1 < my_slabs) load_slab(it + kStages - 1);
    cp_async_commit();

    const int slab0 = t0 + (slab_first + it * slab_step) * kSlab;
    const uint32_t kb = wbase + (it % kStages) * (kFp8 ? C::kStageBytes8 : C::kStageBytes);
    const uint32_t vb = kb + (kFp8 ? C::kSlabBytes8 : C::kSlabBytes);
    // generic pointers to the same fp8 slabs, for the fragment loads
    const uint8_t *k8 = smem + (kb - smem_u32(smem));
    const uint8_t *v8 = k8 + C::kSlabBytes8;
    const int mi = lane >> 3, mr = lane & 7;

    // scores: kMT 16-token m-tiles
    float s[kMT][4];
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) s[mt][e] = 0.f;
      uint4 kx0, kx1;  // fp8: rows lr / lr + 8, 16 bytes = four k-steps' words
#pragma unroll
      for (int ks = 0; ks < kKS; ++ks) {
        uint32_t a[4];
        if (kFp8) {
          if ((ks & 3) == 0) {
            const int r0 = mt * 16 + lr, r1 = r0 + 8;
            kx0 = *reinterpret_cast<const uint4 *>(k8 + swz8<D>(r0, lc + 4 * (ks >> 2)));
            kx1 = *reinterpret_cast<const uint4 *>(k8 + swz8<D>(r1, lc + 4 * (ks >> 2)));
          }
          const int q = ks & 3;
          const uint32_t x0 = q == 0 ? kx0.x : q == 1 ? kx0.y : q == 2 ? kx0.z : kx0.w;
          const uint32_t x1 = q == 0 ? kx1.x : q == 1 ? kx1.y : q == 2 ? kx1.z : kx1.w;
          e4m3x4_to_f16x4(x0, a[0], a[2]);
          e4m3x4_to_f16x4(x1, a[1], a[3]);
          mma_f16_16816(s[mt], a, qf[ks][0], qf[ks][1]);
        } else {
          const int row = mt * 16 + (mi & 1) * 8 + mr;
          ldmatrix_x4(kb + swz<D>(row, ks * 2 + (mi >> 1)), a[0], a[1], a[2], a[3]);
          mma_bf16_16816(s[mt], a, qf[ks][0], qf[ks][1]);
        }
      }
    }
    // scale to log2 units, mask the ragged end of the chunk, tile maximum
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = slab0 + mt * 16 + lr + ((e & 2) ? 8 : 0);
        const float x = j < t1 ? s[mt][e] * score_log2 : -INFINITY;
        s[mt][e] = x;
        if (e & 1)
          mx1 = fmaxf(mx1, x);
        else
          mx0 = fmaxf(mx0, x);
      }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float base0 = mn0 == -INFINITY ? 0.f : mn0;
    const float base1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = fast_exp2(m0 - base0), al1 = fast_exp2(m1 - base1);
    m0 = mn0;
    m1 = mn1;
    float sum0 = 0.f, sum1 = 0.f;
    // P enters the tensor core as two bf16 terms, hi + lo, which together
    // carry 16 significant bits: a single bf16 P (8 bits) alone would add
    // about 1.6e-3 rms relative error to the output. With the fp16 MMAs of
    // the fp8 cache P is one fp16 term (11 bits).
    uint32_t pb[kMT][2], pl[kMT][2];
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) {
      const float p0 = fast_exp2(s[mt][0] - base0), p1 = fast_exp2(s[mt][1] - base1);
      const float p2 = fast_exp2(s[mt][2] - base0), p3 = fast_exp2(s[mt][3] - base1);
      sum0 += p0 + p2;
      sum1 += p1 + p3;
      if (kFp8) {
        pb[mt][0] = movmatrix_trans(pack_f16x2(p0, p1));
        pb[mt][1] = movmatrix_trans(pack_f16x2(p2, p3));
        continue;
      }
      const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
      const uint32_t l01 = pack_bf16x2(p0 - bf16_lo(h01), p1 - bf16_hi(h01));
      const uint32_t l23 = pack_bf16x2(p2 - bf16_lo(h23), p3 - bf16_hi(h23));
      // (token lr, heads 2lc..) -> (head lr, tokens 2lc..): the B fragment of P^T
      pb[mt][0] = movmatrix_trans(h01);
      pb[mt][1] = movmatrix_trans(h23);
      pl[mt][0] = movmatrix_trans(l01);
      pl[mt][1] = movmatrix_trans(l23);
    }
    d0 = d0 * al0 + sum0;
    d1 = d1 * al1 + sum1;
#pragma unroll
    for (int dt = 0; dt < kKS; ++dt) {
      o[dt][0] *= al0;
      o[dt][1] *= al1;
      o[dt][2] *= al0;
      o[dt][3] *= al1;
    }
    // O^T += V^T P^T
    if constexpr (kFp8) {
      // MMA rows lr / lr + 8 of dim tile dt stand for dims (D / 8) lr + 2 dt
      // and + 1: one (D / 8)-byte load per token (tokens t, t+1, t+8, t+9)
      // holds the lane's bytes of every dim tile, paired across tokens with a
      // byte permute (undone when O is stored)
      constexpr int kW = D / 32;  // 32-bit words per token load
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        const int t = mt * 16 + 2 * lc;
        const int byte0 = (D / 8) * lr;
        const int chunk = byte0 >> 4, within = byte0 & 15;
        uint32_t w[4][kW];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int tok = t + (i & 1) + 8 * (i >> 1);
          const uint8_t *src = v8 + swz8<D>(tok, chunk) + within;
          if constexpr (kW == 2) {
            const uint2 x = *reinterpret_cast<const uint2 *>(src);
            w[i][0] = x.x;
            w[i][1] = x.y;
          } else {
            const uint4 x = *reinterpret_cast<const uint4 *>(src);
            w[i][0] = x.x;
            w[i][1] = x.y;
            w[i][2] = x.z;
            w[i][3] = x.w;
          }
        }
#pragma unroll
        for (int dt = 0; dt < kKS; ++dt) {
          uint32_t a[4];
          const unsigned sel = (dt & 1) ? 0x7362u : 0x5140u;
          e4m3x4_to_f16x4(__byte_perm(w[0][dt >> 1], w[1][dt >> 1], sel), a[0], a[1]);
          e4m3x4_to_f16x4(__byte_perm(w[2][dt >> 1], w[3][dt >> 1], sel), a[2], a[3]);
          mma_f16_16816(o[dt], a, pb[mt][0], pb[mt][1]);
        }
      }
    } else
#pragma unroll
    for (int dt = 0; dt < kKS; ++dt)
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        uint32_t a[4];
        {
          const int row = mt * 16 + (mi >> 1) * 8 + mr;
          ldmatrix_x4_trans(vb + swz<D>(row, dt * 2 + (mi & 1)), a[0], a[1], a[2], a[3]);
          mma_bf16_16816(o[dt], a, pb[mt][0], pb[mt][1]);
          mma_bf16_16816(o[dt], a, pl[mt][0], pl[mt][1]);
        }
      }
  }
  cp_async_wait<0>();

#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    d0 += __shfl_xor_sync(0xffffffffu, d0, off);
    d1 += __shfl_xor_sync(0xffffffffu, d1, off);
  }

  // O^T rows lr / lr + 8 of dim tile dt are dims dt*16 + lr / + 8 (bf16),
  // (D / 8) lr + 2 dt / + 1 (fp8)
  auto odim0 = [&](int dt) { return kFp8 ? (D / 8) * lr + 2 * dt : dt * 16 + lr; };
  auto odim1 = [&](int dt) { return kFp8 ? (D / 8) * lr + 2 * dt + 1 : dt * 16 + lr + 8; };

  if constexpr (kPair) {
    // ---- one pair per warp: the state is final; stage it in this warp's
    // own ring memory and write 4 lanes per head, D / 4 dims each ----
    __syncwarp();  // every lane is done with the ring
    float *pm = reinterpret_cast<float *>(smem + warp * kStages *
                                                     (kFp8 ? C::kStageBytes8 : C::kStageBytes));
    float *pd = pm + kMaxGroup;
    float *po = pd + kMaxGroup;  // [8][D]
    if (lr == 0) {
      pm[2 * lc] = m0;
      pm[2 * lc + 1] = m1;
      pd[2 * lc] = d0;
      pd[2 * lc + 1] = d1;
    }
#pragma unroll
    for (int dt = 0; dt < kKS; ++dt) {
      po[(2 * lc) * D + odim0(dt)] = o[dt][0];
      po[(2 * lc + 1) * D + odim0(dt)] = o[dt][1];
      po[(2 * lc) * D + odim1(dt)] = o[dt][2];
      po[(2 * lc + 1) * D + odim1(dt)] = o[dt][3];
    }
    __syncwarp();
    const int hh = lane >> 2;
    constexpr int kPer = D / 4;
    const int c0 = (lane & 3) * kPer;
    if (hh < gt) {
      const float dn = pd[hh];
      const float inv = dn > 0.f ? out_scale / dn : 0.f;
      const size_t row_h = static_cast<size_t>(b) * p.hq + hbase + hh;
#pragma unroll
      for (int q8 = 0; q8 < kPer / 8; ++q8) {
        const float4 x = *reinterpret_cast<const float4 *>(po + hh * D + c0 + 8 * q8);
        const float4 y = *reinterpret_cast<const float4 *>(po + hh * D + c0 + 8 * q8 + 4);
        uint4 v;
        v.x = pack_bf16x2(x.x * inv, x.y * inv);
        v.y = pack_bf16x2(x.z * inv, x.w * inv);
        v.z = pack_bf16x2(y.x * inv, y.y * inv);
        v.w = pack_bf16x2(y.z * inv, y.w * inv);
        *reinterpret_cast<uint4 *>(p.out + row_h * D + c0 + 8 * q8) = v;
      }
      if (p.lse != nullptr && (lane & 3) == 0)
        p.lse[row_h] = dn > 0.f ? (pm[hh] + fast_log2(dn)) * kLn2 : -INFINITY;
    }
    return;
  }

  // ---- combine the 4 warps through shared memory ----
  __syncthreads();  // every warp is done with its ring
  float *sm_m = reinterpret_cast<float *>(smem);          // [4][8]
  float *sm_d = sm_m + kWarps * kMaxGroup;                 // [4][8]
  float *sm_o = sm_d + kWarps * kMaxGroup;                 // [4][8][D]
  if (lr == 0) {
    sm_m[warp * 8 + 2 * lc] = m0;
    sm_m[warp * 8 + 2 * lc + 1] = m1;
    sm_d[warp * 8 + 2 * lc] = d0;
    sm_d[warp * 8 + 2 * lc + 1] = d1;
  }
#pragma unroll
  for (int dt = 0; dt < kKS; ++dt) {
    float *ow = sm_o + warp * kMaxGroup * D;
    ow[(2 * lc) * D + odim0(dt)] = o[dt][0];
    ow[(2 * lc + 1) * D + odim0(dt)] = o[dt][1];
    ow[(2 * lc) * D + odim1(dt)] = o[dt][2];
    ow[(2 * lc + 1) * D + odim1(dt)] = o[dt][3];
  }
  __syncthreads();

  const int tid = threadIdx.x;
  const int hh = tid >> 4;                        // head within the group
  constexpr int kOut = C::kOutPer;                // output dims per thread
  const int c0 = (tid & 15) * kOut;
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w * 8 + hh]);
  const float baseM = M == -INFINITY ? 0.f : M;
  float Dn = 0.f, acc[kOut];
#pragma unroll
  for (int e = 0; e < kOut; ++e) acc[e] = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const float f = fast_exp2(sm_m[w * 8 + hh] - baseM);
    Dn += f * sm_d[w * 8 + hh];
#pragma unroll
    for (int q4 = 0; q4 < kOut / 4; ++q4) {
      const float4 ov =
          *reinterpret_cast<const float4 *>(sm_o + (w * kMaxGroup + hh) * D + c0 + 4 * q4);
      acc[4 * q4] += f * ov.x;
      acc[4 * q4 + 1] += f * ov.y;
      acc[4 * q4 + 2] += f * ov.z;
      acc[4 * q4 + 3] += f * ov.w;
    }
  }
  const float inv = Dn > 0.f ? out_scale / Dn : 0.f;
  // block lse in natural log (-inf when nothing is visible and no sink)
  const float blse = Dn > 0.f ? (M + fast_log2(Dn)) * kLn2 : -INFINITY;
  const bool head_ok = hh < gt;
  const int qh = hbase + hh;
  const size_t row_h = static_cast<size_t>(b) * p.hq + qh;
  // kOut values times `mul` -> bf16 at out[row_h][c0...]
  auto store_out = [&](const float *x, float mul) {
#pragma unroll
    for (int q4 = 0; q4 < kOut / 4; ++q4) {
      uint2 pk;
      pk.x = pack_bf16x2(x[4 * q4] * mul, x[4 * q4 + 1] * mul);
      pk.y = pack_bf16x2(x[4 * q4 + 2] * mul, x[4 * q4 + 3] * mul);
      *reinterpret_cast<uint2 *>(p.out + row_h * D + c0 + 4 * q4) = pk;
    }
  };

  if (nsplit == 1) {
    if (head_ok) {
      store_out(acc, inv);
      if (p.lse != nullptr && (tid & 15) == 0) p.lse[row_h] = blse;
    }
    return;
  }

  const size_t rows_hq = static_cast<size_t>(p.batch) * p.hq;
  if (head_ok) {
#pragma unroll
    for (int q4 = 0; q4 < kOut / 4; ++q4)
      *reinterpret_cast<float4 *>(p.part_o + (split * rows_hq + row_h) * D + c0 + 4 * q4) =
          make_float4(acc[4 * q4] * inv, acc[4 * q4 + 1] * inv, acc[4 * q4 + 2] * inv,
                      acc[4 * q4 + 3] * inv);
    if ((tid & 15) == 0) p.part_lse[split * rows_hq + row_h] = blse;
  }
  __threadfence();
  __syncthreads();
  __shared__ int s_last;
  if (tid == 0) {
    // the counters were zeroed by the kernel launched just before this one,
    // which lets this grid start early: wait for it here, the first use
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const unsigned prev = atomicAdd(p.counters + cidx, 1u);
    s_last = prev == static_cast<unsigned>(nsplit - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- last block: merge the nsplit partials of this (sequence, KV head) ----
  if (head_ok) {
    float Mx = -INFINITY;
    for (int k = 0; k < nsplit; ++k) Mx = fmaxf(Mx, __ldcg(p.part_lse + k * rows_hq + row_h));
    float W = 0.f, r[kOut];
#pragma unroll
    for (int e = 0; e < kOut; ++e) r[e] = 0.f;
    if (Mx != -INFINITY) {
      for (int k = 0; k < nsplit; ++k) {
        const float l = __ldcg(p.part_lse + k * rows_hq + row_h);
        const float w = fast_exp2((l - Mx) * kLog2e);
        if (w == 0.f) continue;
        W += w;
#pragma unroll
        for (int q4 = 0; q4 < kOut / 4; ++q4) {
          const float4 ov = __ldcg(reinterpret_cast<const float4 *>(
              p.part_o + (k * rows_hq + row_h) * D + c0 + 4 * q4));
          r[4 * q4] += w * ov.x;
          r[4 * q4 + 1] += w * ov.y;
          r[4 * q4 + 2] += w * ov.z;
          r[4 * q4 + 3] += w * ov.w;
        }
      }
    }
    store_out(r, W > 0.f ? 1.f / W : 0.f);
    if (p.lse != nullptr && (tid & 15) == 0)
      p.lse[row_h] = W > 0.f ? Mx + fast_log2(W) * kLn2 : -INFINITY;
  }
  if (tid == 0) p.counters[cidx] = 0u;  // ready for the next call / graph replay
}

}  // namespace

DecodePlan plan_decode(int batch, int hq, int hkv, int max_seqlen_k, int window, int num_splits) {
  hkv = hkv * decode_head_tiles(hq, hkv);  // blocks per sequence and split
  int span = window > 0 ? (window < max_seqlen_k ? window : max_seqlen_k) : max_seqlen_k;
  if (span < 1) span = 1;
  long chunk;
  if (num_splits > 0) {
    chunk = (span + num_splits - 1) / num_splits;
  } else {
    // About two blocks per (sequence, KV head) for contexts spread up to
    // `span` (mean taken as span / 2), and at least ~4 waves of two blocks per
    // SM on a 152-SM GB300 for small batches. Measured on GB300 (bf16 and
    // fp8, contiguous and paged): larger blocks cut the per-block prologue and
    // merge traffic; two per pair beat three by 1.5-3%.
    const long pairs = static_cast<long>(batch > 0 ? batch : 1) * (hkv > 0 ? hkv : 1);
    const long est = span / 2 > 0 ? span / 2 : 1;
    long blocks = 2 * pairs;
    if (blocks < 4 * 2 * 152) blocks = 4 * 2 * 152;
    chunk = (pairs * est + blocks - 1) / blocks;
    const long cap = (span + 63) / 64;  // at most 64 splits
    if (chunk < cap) chunk = cap;
  }
  const long unit = kWarps * 32;  // whole warp steps at either head_dim (32 or 16 tokens)
  chunk = (chunk + unit - 1) / unit * unit;
  DecodePlan plan;
  plan.chunk = static_cast<int>(chunk);
  plan.max_splits = static_cast<int>((span + chunk - 1) / chunk);
  if (plan.max_splits < 1) plan.max_splits = 1;
  return plan;
}

DecodeWorkspace decode_workspace_layout(int batch, int hq, int hkv, const DecodePlan &plan,
                                        int head_dim) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  DecodeWorkspace w;
  const size_t rows = static_cast<size_t>(plan.max_splits) * batch * hq;
  w.off_lse = up(rows * head_dim * sizeof(float));
  w.off_counters = w.off_lse + up(rows * sizeof(float));
  w.bytes = w.off_counters + up(static_cast<size_t>(batch) * hkv * decode_head_tiles(hq, hkv) *
                                sizeof(unsigned));
  return w;
}

cudaError_t launch_decode(const DecodeLaunch &a, cudaStream_t stream) {
  Params p;
  p.q = static_cast<const __nv_bfloat16 *>(a.q);
  p.k = static_cast<const __nv_bfloat16 *>(a.k);
  p.v = static_cast<const __nv_bfloat16 *>(a.v);
  p.k8 = static_cast<const uint8_t *>(a.k);
  p.v8 = static_cast<const uint8_t *>(a.v);
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.kv_indptr = a.kv_indptr;
  p.block_table = a.block_table;
  p.seqlens_k = a.seqlens_k;
  p.max_pages = a.max_pages;
  p.page_size = a.page_size;
  p.page_shift = -1;
  if (a.page_size > 0 && (a.page_size & (a.page_size - 1)) == 0) {
    p.page_shift = 0;
    while ((1 << p.page_shift) < a.page_size) ++p.page_shift;
  }
  p.batch = a.batch;
  p.hq = a.hq;
  p.hkv = a.hkv;
  p.group = a.hq / a.hkv;
  p.nht = decode_head_tiles(a.hq, a.hkv);
  p.window = a.window;
  p.chunk = a.plan.chunk;
  p.sinks = a.sinks;
  p.scale_log2 = a.scale * kLog2e;
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.lse = a.lse;
  const DecodeWorkspace w = decode_workspace_layout(a.batch, a.hq, a.hkv, a.plan, a.head_dim);
  uint8_t *ws = static_cast<uint8_t *>(a.workspace);
  p.part_o = reinterpret_cast<float *>(ws);
  p.part_lse = reinterpret_cast<float *>(ws + w.off_lse);
  p.counters = reinterpret_cast<unsigned int *>(ws + w.off_counters);

  // With splits, the merge counters are zeroed by a small kernel that lets
  // the decode grid launch at once (programmatic dependent launch); the decode
  // waits for it only where it first touches a counter, after its K/V pass.
  const bool split = a.plan.max_splits > 1;
  if (split) {
    const int64_t n = static_cast<int64_t>(a.batch) * a.hkv * p.nht;
    const int blocks = static_cast<int>((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
    zero_counters_kernel<<<blocks, 256, 0, stream>>>(p.counters, n);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // Unsplit calls whose visible span is short run one warp per (sequence,
  // KV head); the span bound is the host's, a longer sequence only makes
  // its warp loop longer.
  const int span = a.window > 0 && a.window < a.max_seqlen_k ? a.window : a.max_seqlen_k;
  const bool pair = !split && span <= kPairMaxSpan;
  const dim3 grid = pair ? dim3(static_cast<unsigned>(
                               (static_cast<int64_t>(a.batch) * a.hkv * p.nht + kWarps - 1) /
                               kWarps))
                         : dim3(a.plan.max_splits, a.hkv * p.nht, a.batch);
  auto go = [&](auto kernel, int smem) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = split ? 1 : 0;
    cudaLaunchKernelEx(&cfg, kernel, p);
  };
  const bool paged = a.block_table != nullptr;
  auto pick2 = [&](auto dim, auto one_pair) {
    constexpr int D = decltype(dim)::value;
    constexpr bool P = decltype(one_pair)::value;
    if (a.fp8) {
      if (paged)
        go(decode_kernel<D, true, true, P>, Ring<D, true, true, P>::kSmemBytes);
      else
        go(decode_kernel<D, false, true, P>, Ring<D, false, true, P>::kSmemBytes);
    } else {
      if (paged)
        go(decode_kernel<D, true, false, P>, Ring<D, true, false, P>::kSmemBytes);
      else
        go(decode_kernel<D, false, false, P>, Ring<D, false, false, P>::kSmemBytes);
    }
  };
  auto pick = [&](auto dim) {
    if (pair)
      pick2(dim, std::true_type());
    else
      pick2(dim, std::false_type());
  };
  if (a.head_dim == 128)
    pick(std::integral_constant<int, 128>());
  else
    pick(std::integral_constant<int, 64>());
  return cudaGetLastError();
}

}  // namespace sinkattn

// ---------------------------------------------------------------------------
// Allocation-free decode entry point.
//
// Some callers cannot hand the library a scratch buffer: code that runs under
// a memory planner owning every device byte, plugin hosts that forbid
// allocation while enqueueing work, and latency-critical loops where
// cudaMalloc/cudaFree may synchronise the device. For them,
// sinkattn_decode_noalloc keeps the split-KV partials and the block counters
// in the fixed array below instead of a caller workspace. The array is part
// of the library image: every GPU that loads the library holds it until the
// process exits. All calls on a device share it and it keeps the previous
// call's contents; the counters are cleared on the stream at the start of
// each call and the partials are always written before they are read. Two
// calls whose kernels overlap on the GPU (different streams, no ordering
// between them) race on this array and give wrong results.

namespace sinkattn {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SINKATTN_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch in the calling thread's current
// context, looked up once per context with that context's device current (the
// host-side symbol is not a device address). The cache is keyed by the
// driver's context id, which is never reused within a process, so a context
// created after cudaDeviceReset (where the module, and so the array, may sit
// at another address) gets a fresh lookup.
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// *id = the current context's id, or 0 when no context is current yet.
cudaError_t current_context_id(unsigned long long *id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  if (get_current == nullptr || get_id == nullptr) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  *id = 0;
  if (ctx != nullptr && get_id(ctx, id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  return cudaSuccess;
}

cudaError_t noalloc_scratch(void **ptr) {
  static std::mutex mu;
  static unsigned long long ids[64] = {};
  static void *addr[64] = {};
  static int used = 0, next = 0;
  std::lock_guard<std::mutex> lock(mu);
  unsigned long long id = 0;
  cudaError_t e = current_context_id(&id);
  if (e != cudaSuccess) return e;
  for (int i = 0; id != 0 && i < used; ++i)
    if (ids[i] == id) {
      *ptr = addr[i];
      return cudaSuccess;
    }
  // The lookup makes the current device's primary context current if no
  // context was, so the id is read again after it.
  void *p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e == cudaSuccess) e = current_context_id(&id);
  if (e != cudaSuccess) return e;
  if (id == 0) return cudaErrorDeviceUninitialized;
  const int slot = used < 64 ? used++ : (next++ & 63);  // past 64 contexts, recycle entries
  ids[slot] = id;
  addr[slot] = p;
  *ptr = p;
  return cudaSuccess;
}

bool is_aligned(const void *p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

}  // namespace
}  // namespace sinkattn

extern "C" sinkattn_status_t sinkattn_decode_noalloc(
    const void *q, const void *k_cache, const void *v_cache, const int32_t *kv_indptr,
    const int32_t *block_table, const int32_t *seqlens_k, int64_t kv_rows, int max_pages_per_seq,
    int page_size, int batch, int max_seqlen_k, int hq, int hkv, int head_dim, const float *sinks,
    sinkattn_mask_t mask, int num_splits, void *out, float *lse, void *stream) {
  using namespace sinkattn;
  if (batch < 0 || max_seqlen_k < 0 || hq <= 0 || hkv <= 0 || hq % hkv != 0 || num_splits < 0 ||
      kv_rows < 0 || mask.window < 0 || !isfinite(mask.scale) || !(mask.scale > 0.f))
    return SINKATTN_ERR_INVALID_ARGUMENT;
  if (!decode_head_dim_ok(head_dim)) return SINKATTN_ERR_UNSUPPORTED;
  const bool paged = block_table != nullptr;
  if (paged == (kv_indptr != nullptr)) return SINKATTN_ERR_INVALID_ARGUMENT;
  if (paged && (seqlens_k == nullptr || page_size <= 0 || max_pages_per_seq <= 0))
    return SINKATTN_ERR_INVALID_ARGUMENT;
  if (!paged && seqlens_k != nullptr) return SINKATTN_ERR_INVALID_ARGUMENT;
  if (batch == 0) return SINKATTN_OK;
  if (!q || !k_cache || !v_cache || !out) return SINKATTN_ERR_INVALID_ARGUMENT;
  if (!is_aligned(q, 16) || !is_aligned(k_cache, 16) || !is_aligned(v_cache, 16) ||
      !is_aligned(out, 16) || (kv_indptr && !is_aligned(kv_indptr, 4)) ||
      (block_table && !is_aligned(block_table, 4)) || (seqlens_k && !is_aligned(seqlens_k, 4)) ||
      (sinks && !is_aligned(sinks, 4)) || (lse && !is_aligned(lse, 4)))
    return SINKATTN_ERR_INVALID_ARGUMENT;
  if (batch > 65535 || static_cast<int64_t>(hkv) * decode_head_tiles(hq, hkv) > 65535)
    return SINKATTN_ERR_UNSUPPORTED;
  const DecodePlan plan = plan_decode(batch, hq, hkv, max_seqlen_k, mask.window, num_splits);
  // the plan's scratch must fit the fixed array
  if (plan.max_splits > 1 &&
      decode_workspace_layout(batch, hq, hkv, plan, head_dim).bytes >
          SINKATTN_NOALLOC_SCRATCH_BYTES)
    return SINKATTN_ERR_WORKSPACE_TOO_SMALL;
  void *scratch = nullptr;
  const cudaError_t se = noalloc_scratch(&scratch);
  if (se != cudaSuccess) return static_cast<sinkattn_status_t>(cuda_status(se));
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
  a.workspace = scratch;
  a.plan = plan;
  a.head_dim = head_dim;
  return static_cast<sinkattn_status_t>(cuda_status(launch_decode(a, static_cast<cudaStream_t>(stream))));
}
