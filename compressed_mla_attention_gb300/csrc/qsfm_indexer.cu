// Lightning-indexer top-k (QuantLightningIndexerV2, quant mode 1) for sm_103a.
//
// For every query token: score_j = sum_h W[h] ReLU(Sq[h] Sk[j] (Q[h] . K[j]))
// over the keys it may see, then the topk keys of largest score
// (QuantLightningIndexerV2, "功能说明": the formula and its three steps).
//
// Two kernels on one stream.
//
// ix_score_kernel, one CTA per SM. The query tokens of a batch are taken in
// rows of up to G consecutive tokens (G x heads rounded up to 16 <= 256, the
// largest MMA N), a row's keys in 128-key tiles (one paged block each). The
// tiles of all rows, laid end to end, are cut into equal contiguous ranges,
// one per CTA, so every SM streams the same number of key bytes whatever the
// mix of sequence lengths, and each key block is read once for all the
// tokens of its row. Per tile:
//   * TMA brings the key block (128 rows x 128 bytes, 128-byte swizzle) into
//     one of as many stages as shared memory holds (11 for two tokens of 64
//     heads; freed by the MMAs) and a bulk copy its 128 key scales into one
//     of 16 scale slots (freed by the epilogue);
//   * S^T[j, (g, h)] = K[j] . Q[g, h] for all the row's tokens at once:
//     tcgen05.mma kind::f8f6f4 (e4m3 x e4m3, fp32 accumulate), M = 128 keys,
//     N = G x padded heads, four MMAs of K = 32, into one of two TMEM
//     accumulators. The row's Q arrives as one 3-D TMA box (heads past the
//     real ones zero-filled), double-buffered so the next row's Q lands
//     while this row computes;
//   * 16 epilogue warps in four groups read S^T (one thread per key) and
//     reduce each token's heads to the key's score, stored to that token's
//     fp32 score row in the workspace; the groups take the (tile, token)
//     items in turn, and up to 4 accumulators let the MMAs run ahead.
// Roles: warp 0 TMA producer, warp 1 MMA issue, warps 2-17 epilogue.
//
// ix_select_kernel, one CTA per query token, launched with programmatic
// serialization so its launch overlaps the score kernel's tail. It loads the
// token's scores into registers as order-preserving 32-bit keys and finds
// the k-th largest by a radix select whose first digit starts at the
// highest bit where the largest key and a lower bound of the k-th largest
// differ (keys below the bound are never counted, and the digits resolve the
// upper tail where the threshold lies). It writes the selected keys in
// ascending order (equal scores: the smaller key first), then -1.
//
// Every mbarrier wait is bounded (timeout -> fault bit, abort flag, orderly
// exit).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "qsfm_device.cuh"
#include "qsfm_internal.h"

namespace qsfm {
namespace {

constexpr int kIxThreads = 576;  // warp 0 producer, warp 1 MMA, warps 2-17 epilogue
constexpr int kIxEpiWarps = 16;
constexpr int kIxGroups = kIxEpiWarps / 4;
constexpr int kIxDim = 128;        // bytes (= e4m3 elements) per query / key row
constexpr int kIxTile = 128;       // keys per tile (one paged block)
constexpr int kIxMaxStages = 12;  // key stages (as many as shared memory holds)
constexpr int kIxSSlots = 16;      // key-scale ring (freed by the epilogue, which trails the MMAs)
static_assert(kIxSSlots == 16, "scale slots and their phases are taken from the low bits of the tile count");
constexpr int kIxMaxKeys = 32768;  // keys per token the select holds in shared memory
constexpr int kIxMaxHeads = 64;
constexpr int kIxMaxN = 256;       // MMA N = tokens of a row x padded heads
constexpr int kIxMaxG = 16;        // tokens per row (16 padded heads each)
constexpr uint64_t kIxTimeoutNs = 2000000000ull;

// score kernel shared memory (byte offsets from a 1024-aligned base): a
// fixed region, then two Q slots of x.qslot bytes, then x.stages key stages
constexpr uint32_t kXKs = 0;                                    // [scale slot][128] f32 key scales
constexpr uint32_t kXCw = kXKs + kIxSSlots * kIxTile * 4;       // [2][256] f32 W * Sq
constexpr uint32_t kXRow = kXCw + 2 * kIxMaxN * 4;              // [2][32] i32: nvis per token, flag
constexpr uint32_t kXValid = kXRow + 2 * 32 * 4;                // [scale slot] i32: -1 bad block, else 0 / first key row
constexpr uint32_t kXScan = kXValid + kIxSSlots * 4;            // [64] i32 scan scratch
constexpr uint32_t kXBar = kXScan + 256;                        // barriers, tmem slot, flags, plan
constexpr uint32_t kXFixed = (kXBar + 640 + 1023) & ~1023u;     // the Q slots start here
constexpr uint32_t kXSmemMax = 232448;                          // dynamic shared memory of a CTA
constexpr uint32_t kXStage = kIxTile * kIxDim;                  // 16 KB key stage

// barriers: key stage full / empty, accumulator full / empty (up to 4
// accumulators), Q slot full / empty, head factors of a slot published,
// key-scale slot full / empty, drain
constexpr int kIxMaxAcc = 4;
constexpr int kXbFull = 0, kXbEmpty = kIxMaxStages, kXbTFull = 2 * kIxMaxStages, kXbTEmpty = kXbTFull + kIxMaxAcc,
              kXbQFull = kXbTEmpty + kIxMaxAcc, kXbQEmpty = kXbQFull + 2, kXbCwFull = kXbQEmpty + 2,
              kXbSFull = kXbCwFull + 2, kXbSEmpty = kXbSFull + kIxSSlots, kXbDrain = kXbSEmpty + kIxSSlots,
              kXbCount = kXbDrain + 1;
static_assert(kXbCount * 8 <= 576, "barriers overlap the tmem slot");

struct IxSmem {
  uint32_t base;
  uint8_t* ptr;
  __device__ uint64_t* bar(int i) const { return reinterpret_cast<uint64_t*>(ptr + kXBar) + i; }
  __device__ uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(ptr + kXBar + 576); }
  __device__ volatile int* abort_flag() const { return reinterpret_cast<volatile int*>(ptr + kXBar + 584); }
  __device__ int* plan() const { return reinterpret_cast<int*>(ptr + kXBar + 592); }
  __device__ float* f(uint32_t off) const { return reinterpret_cast<float*>(ptr + off); }
  __device__ int* i(uint32_t off) const { return reinterpret_cast<int*>(ptr + off); }
};

__device__ __forceinline__ bool ix_wait(const IxSmem& sm, int bar, uint32_t parity, int* fault) {
  if (mbar_wait_bounded(sm.bar(bar), parity, sm.abort_flag(), kIxTimeoutNs)) return true;
  if (!*sm.abort_flag()) {
    *sm.abort_flag() = 1;
    atomicOr(fault, QSFM_FAULT_TIMEOUT);
  }
  return false;
}

// lane 0 waits, the warp follows (a timeout is seen by every lane)
__device__ __forceinline__ bool ix_warp_wait(const IxSmem& sm, int bar, uint32_t parity, int* fault) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = ix_wait(sm, bar, parity, fault);
  __syncwarp();
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// L2 policy for data read once (the key blocks and their scales): evicted
// first, so the streamed keys do not push the score rows out of L2 before
// the select kernel reads them.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 2-D tiled TMA load with an L2 cache policy.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const void* tmap, int x, int y, uint64_t* bar,
                                                 uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// 1-D bulk copy global -> shared with an L2 cache policy, completing on
// `bar` (both addresses and the size multiples of 16 bytes).
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mma_f8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// Batch b, position s, chunk length s1 and rows in use s1e (seqused_q) of
// query token t.
__device__ __forceinline__ void ix_token(const qsfm_indexer_params& p, int t, int& b, int& s, int& s1, int& s1e) {
  if (p.layout_q == QSFM_LAYOUT_BSND) {
    b = t / p.max_s1;
    s = t - b * p.max_s1;
    s1 = p.max_s1;
  } else {
    int lo = 0, hi = p.batch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(p.cu_seqlens_q + mid) <= t) lo = mid; else hi = mid - 1;
    }
    b = lo;
    const int c0 = __ldg(p.cu_seqlens_q + b);
    s = t - c0;
    s1 = __ldg(p.cu_seqlens_q + b + 1) - c0;
  }
  s1e = p.seqused_q != nullptr ? min(s1, __ldg(p.seqused_q + b)) : s1;
}

// Keys of batch b: seqused_k[b] (paged; BSND, max_sk without seqused_k) or
// the cu_seqlens_k difference (TND), never past the end of a TND key tensor.
__device__ __forceinline__ int ix_keys(const qsfm_indexer_params& p, int b) {
  if (p.layout_k == QSFM_LAYOUT_KV_TND) {
    const int c0 = __ldg(p.cu_seqlens_k + b), c1 = __ldg(p.cu_seqlens_k + b + 1);
    return (c0 < 0 || c0 > p.total_k) ? 0 : max(0, min(c1, p.total_k) - c0);
  }
  if (p.layout_k == QSFM_LAYOUT_KV_BSND && p.seqused_k == nullptr) return p.max_sk;
  return __ldg(p.seqused_k + b);
}

// Key tensor row of batch b's key 0 (BSND, TND; paged keys go through the
// block table).
__device__ __forceinline__ long long ix_key_base(const qsfm_indexer_params& p, int b) {
  return p.layout_k == QSFM_LAYOUT_KV_TND ? (long long)__ldg(p.cu_seqlens_k + b) : (long long)b * p.max_sk;
}

// Keys the token at position s of batch b (chunk length s1) may see: all
// its batch's keys (mask_mode 0), or the compressed keys whose last
// original token is at or before p_c (mask_mode 3). Not capped.
__device__ __forceinline__ int ix_visible(const qsfm_indexer_params& p, int b, int s, int s1) {
  const int sk = ix_keys(p, b);
  if (p.mask_mode == 0) return sk;
  const int r = p.cmp_ratio;
  const int res = p.cmp_residual_k != nullptr ? __ldg(p.cmp_residual_k + b) : 0;
  const int pc = sk * r + res - s1 + s;
  return max(0, min(sk, div_floor(pc + 1, r)));
}

// The row that starts at token t: its batch b, tokens g (0 when no row
// starts at t) and tiles. Rows start at positions 0, G, 2G ... of the rows
// in use; the last token of a row sees the most keys (p_c grows with s).
__device__ __forceinline__ int ix_row(const qsfm_indexer_params& p, int t, int gmax, int kcap, int& b, int& g) {
  int s, s1, s1e;
  ix_token(p, t, b, s, s1, s1e);
  if (s >= s1e || s % gmax != 0) {
    g = 0;
    return 0;
  }
  g = min(gmax, s1e - s);
  const int nv = min(kcap, ix_visible(p, b, s + g - 1, s1));
  return (nv + kIxTile - 1) / kIxTile;
}

// A CTA's walk over the rows that hold tiles: row start token t, its batch,
// tokens and tiles, and the global index of its first tile.
struct IxWalk {
  int t, b, g, tiles, start;
};

// Advance to the next row with tiles; false past the last token.
__device__ __forceinline__ bool ix_next(const qsfm_indexer_params& p, int T, int gmax, int kcap, IxWalk& w) {
  w.start += w.tiles;
  int t = w.t + max(w.g, 1);
  while (t < T) {
    int b, g;
    const int tiles = ix_row(p, t, gmax, kcap, b, g);
    if (tiles > 0) {
      w.t = t;
      w.b = b;
      w.g = g;
      w.tiles = tiles;
      return true;
    }
    t += max(g, 1);
  }
  return false;
}

// Order-preserving 32-bit key of a score (-0 taken as +0 by adding +0):
// non-negative scores get the sign bit set, negative ones are inverted.
__device__ __forceinline__ uint32_t score_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.f);
  return u ^ (uint32_t(int32_t(u) >> 31) | 0x80000000u);
}

// Exclusive prefix sum of v over the block's NT threads (scratch: 64 ints),
// the total in `total`.
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int tid, int* scratch, int& total) {
  constexpr int kW = NT / 32;
  const int lane = tid & 31, warp = tid >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kW ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += u;
    }
    if (lane < kW) scratch[32 + lane] = w;
  }
  __syncthreads();
  total = scratch[32 + kW - 1];
  const int r = (warp ? scratch[32 + warp - 1] : 0) + incl - v;
  __syncthreads();  // scratch is reused by the next call
  return r;
}

// Shape of a launch of the score kernel.
struct IxShape {
  int T;        // query tokens
  int gmax;     // tokens per row at most
  int hp;       // heads rounded up to 16
  int kcap;     // keys per token at most
  int kstride;  // floats per token's score row in the workspace
  int nacc;     // TMEM columns of one accumulator (gmax * hp rounded up to 32)
  int na;       // accumulators (4 when they fit in 512 columns, else 2)
  int tcols;    // TMEM columns allocated (a power of two >= na * nacc)
  int qslot;    // bytes of a Q slot (gmax * hp * 128 rounded up to 1024)
  int stages;   // key stages
  int paged;    // keys paged through the block table (else BSND / TND rows)
  __host__ __device__ uint32_t q_off(int slot) const { return kXFixed + uint32_t(slot) * uint32_t(qslot); }
  __host__ __device__ uint32_t key_off(uint32_t st) const { return kXFixed + 2u * uint32_t(qslot) + st * kXStage; }
  __host__ __device__ uint32_t smem_bytes() const { return key_off(uint32_t(stages)) + 1024; }
};

// ------------------------------------------------------------- producer
// The head factors W * Sq of row w's tokens (0 past the real heads), the
// keys each token sees and whether any query scale is negative, into Q slot
// `slot`'s shared tables; all 32 lanes of the calling warp arrive on the
// slot's CwFull barrier.
__device__ __forceinline__ void ix_publish(const qsfm_indexer_params& p, const IxShape& x, const IxSmem& sm,
                                           const IxWalk& w, int slot) {
  const int lane = threadIdx.x & 31;
  float* cwb = sm.f(kXCw);
  int* rowi = sm.i(kXRow);
  bool neg = false;  // a negative query scale (not produced by amax / 448 quantisation)
  for (int i = lane; i < w.g * x.hp; i += 32) {
    const int gg = i / x.hp, h = i - gg * x.hp;
    float c = 0.f;
    if (h < p.heads) {
      const size_t o = size_t(w.t + gg) * p.heads + h;
      const float sq = __ldg(p.query_scale + o);
      c = __ldg(p.weights + o) * sq;
      neg |= sq < 0.f;
    }
    cwb[slot * kIxMaxN + i] = c;
  }
  if (lane < w.g) {
    int b, s, s1, s1e;
    ix_token(p, w.t + lane, b, s, s1, s1e);
    rowi[slot * 32 + lane] = min(x.kcap, ix_visible(p, b, s, s1));
  }
  const bool any_neg = __any_sync(0xffffffffu, neg);
  if (lane == 0) rowi[slot * 32 + kIxMaxG] = any_neg ? 1 : 0;
  mbar_arrive(sm.bar(kXbCwFull + slot));
}

// Per row: the row's Q (one 3-D box: hp heads x gmax tokens), then the row's
// key tiles in this CTA's range (the block table read 32 entries at a time;
// per tile the key block into a stage and its scales into a scale slot).
// Once the first stages are in flight, the row's head factors W * Sq and the
// keys each token sees are published for the epilogue (the first row's by
// an epilogue warp, at the start).
__device__ void ix_produce(const qsfm_indexer_params& p, const IxShape& x, const IxSmem& sm, IxWalk w, int lo,
                           int hi, int* fault, const CUtensorMap* kmap, const CUtensorMap* qmap) {
  const int lane = threadIdx.x & 31;
  int* valid = sm.i(kXValid);
  const uint32_t qbytes = uint32_t(x.gmax * x.hp * kIxDim);
  const uint64_t pol = l2_evict_first();
  // tile n's stage and scale slot, and the parities of their previous use,
  // kept as running counters (no divisions on the issuing lane)
  const uint32_t ns = uint32_t(x.stages);
  const uint32_t key0 = sm.base + x.key_off(0);
  uint32_t n = 0, st = 0, st_par = 1;
  for (uint32_t qn = 0;; ++qn) {
    const int slot = int(qn & 1);
    if (qn >= 2 && !ix_warp_wait(sm, kXbQEmpty + slot, ((qn >> 1) & 1) ^ 1, fault)) return;
    if (lane == 0) {
      mbar_arrive_expect_tx(sm.bar(kXbQFull + slot), qbytes);
      tma_load_3d(sm.base + x.q_off(slot), qmap, 0, 0, w.t, sm.bar(kXbQFull + slot));
    }
    // the first row's tables are published by an epilogue warp at the start
    // (idle then); later rows' by this warp once their first stages are in
    // flight
    const int i_lo = max(lo - w.start, 0), i_hi = min(hi - w.start, w.tiles);
    const int i_pub = i_lo + min(x.stages, i_hi - i_lo);
    bool published = qn == 0;
    const long long kbase = x.paged ? 0 : ix_key_base(p, w.b);  // BSND / TND: batch b's key 0
    for (int i0 = i_lo; i0 < i_hi; i0 += 32) {
      int mine = -1;
      if (x.paged && i0 + lane < i_hi) mine = __ldg(p.block_table + size_t(w.b) * p.max_blocks + i0 + lane);
      const int i1 = min(i_hi, i0 + 32);
      for (int i = i0; i < i1; ++i, ++n) {
        if (i == i_pub && !published) {
          ix_publish(p, x, sm, w, slot);
          published = true;
        }
        const int blk = __shfl_sync(0xffffffffu, mine, i - i0);
        bool go = true;
        const uint32_t ss = n & (kIxSSlots - 1), ss_par = ((n >> 4) & 1) ^ 1;
        if (lane == 0) {
          if ((n >= ns && !ix_wait(sm, kXbEmpty + st, st_par, fault)) ||
              (n >= kIxSSlots && !ix_wait(sm, kXbSEmpty + ss, ss_par, fault))) {
            go = false;
          } else if (!x.paged) {
            // BSND / TND rows: the box may run past the batch or the tensor
            // (zero fill, scores masked); the epilogue reads the scales
            const int row0 = int(kbase) + i * kIxTile;
            valid[ss] = row0;
            mbar_arrive_expect_tx(sm.bar(kXbFull + st), kIxTile * kIxDim);
            tma_load_2d_hint(key0 + st * kXStage, kmap, 0, row0, sm.bar(kXbFull + st), pol);
            mbar_arrive(sm.bar(kXbSFull + ss));
          } else if (blk < 0 || blk >= p.num_blocks) {
            atomicOr(fault, QSFM_FAULT_CMP_BLOCK_ID);
            valid[ss] = -1;  // the tile's scores become -inf; nothing is read
            mbar_arrive(sm.bar(kXbFull + st));
            mbar_arrive(sm.bar(kXbSFull + ss));
          } else {
            valid[ss] = 0;
            mbar_arrive_expect_tx(sm.bar(kXbFull + st), kIxTile * kIxDim);
            tma_load_2d_hint(key0 + st * kXStage, kmap, 0, blk * kIxTile, sm.bar(kXbFull + st), pol);
            mbar_arrive_expect_tx(sm.bar(kXbSFull + ss), kIxTile * 4);
            bulk_g2s_hint(sm.base + kXKs + ss * (kIxTile * 4), p.key_scale + size_t(blk) * kIxTile, kIxTile * 4,
                          sm.bar(kXbSFull + ss), pol);
          }
        }
        if (__shfl_sync(0xffffffffu, go ? 1 : 0, 0) == 0) return;
        if (++st == ns) {
          st = 0;
          st_par ^= 1;
        }
      }
    }
    if (!published) ix_publish(p, x, sm, w, slot);
    if (!ix_next(p, x.T, x.gmax, x.kcap, w) || w.start >= hi) return;
  }
}

// ------------------------------------------------------------- MMA issue
// One thread. Per tile: S^T = K Q^T for the row's g tokens (N = g * hp) into
// accumulator n mod na; the row's Q slot is released after its last tile.
__device__ void ix_mma(const qsfm_indexer_params& p, const IxShape& x, const IxSmem& sm, IxWalk w, int lo, int hi,
                       uint32_t tmem, int* fault) {
  const uint32_t na = uint32_t(x.na), ns = uint32_t(x.stages), nacc = uint32_t(x.nacc);
  const uint64_t kdesc0 = make_sdesc_sw128(sm.base + x.key_off(0), 16, 1024);
  // tile n's stage and accumulator with the parities of their use, kept as
  // running counters (no divisions on the issuing thread)
  uint32_t n = 0, st = 0, st_par = 0, a = 0, a_par = 0;
  for (uint32_t qn = 0;; ++qn) {
    const int slot = int(qn & 1);
    if (!ix_wait(sm, kXbQFull + slot, (qn >> 1) & 1, fault)) return;
    // e4m3 x e4m3 (format code 0 for A and B), fp32 accumulate, both K-major
    const uint32_t idesc = make_idesc_bf16(128, w.g * x.hp, 0, 0, true);
    const uint64_t bdesc = make_sdesc_sw128(sm.base + x.q_off(slot), 16, 1024);
    const int i_lo = max(lo - w.start, 0), i_hi = min(hi - w.start, w.tiles);
    for (int i = i_lo; i < i_hi; ++i, ++n) {
      if (!ix_wait(sm, kXbFull + st, st_par, fault)) return;
      if (n >= na && !ix_wait(sm, kXbTEmpty + a, a_par ^ 1, fault)) return;
      tc_fence_after();
      const uint64_t adesc = kdesc0 + uint64_t((st * kXStage) >> 4);
      const uint32_t d = tmem + a * nacc;
#pragma unroll
      for (int k = 0; k < kIxDim / 32; ++k)  // 32 e4m3 (32 bytes) of d per MMA
        mma_f8(d, adesc + uint64_t((k * 32) >> 4), bdesc + uint64_t((k * 32) >> 4), idesc, k > 0 ? 1u : 0u);
      mma_commit(sm.bar(kXbTFull + a));
      mma_commit(sm.bar(kXbEmpty + st));
      if (++st == ns) {
        st = 0;
        st_par ^= 1;
      }
      if (++a == na) {
        a = 0;
        a_par ^= 1;
      }
    }
    mma_commit(sm.bar(kXbQEmpty + slot));
    if (!ix_next(p, x.T, x.gmax, x.kcap, w) || w.start >= hi) return;
  }
}

// (s0, s1) += (c0, c1) * (r0, r1): two fp32 FMAs in one packed instruction
// (each lane rounds as fmaf does).
__device__ __forceinline__ void fma2(float& s0, float& s1, float c0, float c1, float r0, float r1) {
  asm("{\n .reg .b64 a, b, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n mov.b64 d, {%0, %1};\n"
      " fma.rn.f32x2 d, a, b, d;\n mov.b64 {%0, %1}, d;\n}"
      : "+f"(s0), "+f"(s1)
      : "f"(c0), "f"(c1), "f"(r0), "f"(r1));
}

// Score of one key for one token from its hp accumulator columns at taddr:
// with non-negative scales W ReLU(Sq Sk x) = Sk (W Sq) ReLU(x), the head
// factors cw = W * Sq (0 past the real heads, whose columns hold 0 from the
// zero-filled Q rows); otherwise the formula as written.
__device__ __forceinline__ float ix_key_score(const qsfm_indexer_params& p, uint32_t taddr, int hp, const float* cw,
                                              bool fast, float sk, int t) {
  const float* W = p.weights + size_t(t) * p.heads;
  const float* Sq = p.query_scale + size_t(t) * p.heads;
  if (hp == kIxMaxHeads) {  // two halves of 32 columns
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f, acc = 0.f;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float v[32];
      tmem_ld32(taddr + 32 * half, v);
      tmem_ld_wait();
      if (fast) {
        const float4* c4 = reinterpret_cast<const float4*>(cw + 32 * half);
#pragma unroll
        for (int h = 0; h < 32; h += 4) {
          const float4 c = c4[h >> 2];
          fma2(s0, s1, c.x, c.y, fmaxf(0.f, v[h]), fmaxf(0.f, v[h + 1]));
          fma2(s2, s3, c.z, c.w, fmaxf(0.f, v[h + 2]), fmaxf(0.f, v[h + 3]));
        }
      } else {
#pragma unroll
        for (int h = 0; h < 32; ++h)
          if (32 * half + h < p.heads)
            acc += __ldg(W + 32 * half + h) * fmaxf(0.f, (__ldg(Sq + 32 * half + h) * sk) * v[h]);
      }
    }
    return fast ? sk * ((s0 + s1) + (s2 + s3)) : acc;
  }
  float s0 = 0.f, acc = 0.f;
  for (int c = 0; c < hp; c += 16) {
    float v[16];
    tmem_ld16(taddr + uint32_t(c), v);
    tmem_ld_wait();
    if (fast) {
#pragma unroll
      for (int h = 0; h < 16; ++h) s0 = fmaf(cw[c + h], fmaxf(0.f, v[h]), s0);
    } else {
#pragma unroll
      for (int h = 0; h < 16; ++h)
        if (c + h < p.heads) acc += __ldg(W + c + h) * fmaxf(0.f, (__ldg(Sq + c + h) * sk) * v[h]);
    }
  }
  return fast ? sk * s0 : acc;
}

// ------------------------------------------------------------- epilogue
// Warps 2-17 in four groups of 4; warp w reads TMEM lanes 32 (w mod 4) ..
// + 31, its key rows. Every warp visits every tile; the (tile n, token gg)
// items go to the groups in turn (to group (n g + gg) mod 4), so the
// groups share the tiles' tokens evenly whatever the tokens per row.
__device__ void ix_epilogue(const qsfm_indexer_params& p, const IxShape& x, const IxSmem& sm, IxWalk w, int lo,
                            int hi, uint32_t tmem, float* ws, int* fault) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3, grp = (warp - 2) >> 2;
  const int row = 32 * quarter + lane;
  const uint32_t na = uint32_t(x.na), nacc = uint32_t(x.nacc);
  const float* cwb = sm.f(kXCw);
  const int* rowi = sm.i(kXRow);
  const float* ksm = sm.f(kXKs);
  const int* valid = sm.i(kXValid);
  uint32_t n = 0, a = 0, a_par = 0;  // tile n's accumulator and the parity of its use
  if (warp == 2) ix_publish(p, x, sm, w, 0);  // the first row's tables (the producer publishes the rest)
  for (uint32_t qn = 0;; ++qn) {
    const int slot = int(qn & 1);
    if (!ix_warp_wait(sm, kXbCwFull + slot, (qn >> 1) & 1, fault)) return;
    const bool neg = rowi[slot * 32 + kIxMaxG] != 0;
    const int i_lo = max(lo - w.start, 0), i_hi = min(hi - w.start, w.tiles);
    for (int i = i_lo; i < i_hi; ++i, ++n) {
      const uint32_t ss = n & (kIxSSlots - 1);
      // this group's first item of the tile: gg = grp - n g (mod 4)
      const int first = int((uint32_t(grp) - n * uint32_t(w.g)) & uint32_t(kIxGroups - 1));
      if (!ix_warp_wait(sm, kXbTFull + a, a_par, fault)) return;
      float sk = 0.f;
      int ok = 0;
      if (first < w.g) {
        if (!ix_warp_wait(sm, kXbSFull + ss, (n >> 4) & 1, fault)) return;  // the scales landed
        const int v0 = valid[ss];  // -1: a bad block; else 0 (paged) or the tile's first key row
        ok = v0 >= 0;
        if (x.paged) {
          sk = ksm[ss * kIxTile + row];
        } else if (ok && i * kIxTile + row < rowi[slot * 32 + w.g - 1]) {  // the row's keys (its last token sees most)
          sk = __ldg(p.key_scale + v0 + row);
        }
      }
      tc_fence_after();
      __syncwarp();
      // the scale slot may be refilled (tile n's accumulator being full, the
      // producer has already seen the slot's previous use released)
      if (lane == 0) mbar_arrive(sm.bar(kXbSEmpty + ss));
      const int j = i * kIxTile + row, jw = i * kIxTile + 32 * quarter;
      const uint32_t taddr = tmem + a * nacc + (uint32_t(32 * quarter) << 16);
      const bool fast = __all_sync(0xffffffffu, !neg && sk >= 0.f);
      for (int gg = first; gg < w.g; gg += kIxGroups) {
        const int nv = rowi[slot * 32 + gg];
        if (jw >= nv) continue;  // the warp's 32 keys are all past this token's
        const float sc = ix_key_score(p, taddr + uint32_t(gg * x.hp), x.hp, cwb + slot * kIxMaxN + gg * x.hp, fast,
                                      sk, w.t + gg);
        if (j < nv) ws[size_t(w.t + gg) * x.kstride + j] = ok ? sc : -INFINITY;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.bar(kXbTEmpty + a));
      if (++a == na) {
        a = 0;
        a_par ^= 1;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.bar(kXbQEmpty + slot));
    if (!ix_next(p, x.T, x.gmax, x.kcap, w) || w.start >= hi) return;
  }
}

// ------------------------------------------------------------- score kernel
__global__ void __maxnreg__(96)
    ix_score_kernel(const qsfm_indexer_params p, const IxShape x, float* ws, int* fault,
                    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  IxSmem sm;
  sm.base = (raw + 1023u) & ~1023u;
  sm.ptr = smem_raw + (sm.base - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t tcols = uint32_t(x.tcols);
  grid_launch_dependents();  // the select kernel may be scheduled as CTAs finish
  if (tid == 0) {
    for (int i = 0; i < x.stages; ++i) {
      mbar_init(sm.bar(kXbFull + i), 1);
      mbar_init(sm.bar(kXbEmpty + i), 1);  // the MMAs' commit
    }
    for (int i = 0; i < kIxSSlots; ++i) {
      mbar_init(sm.bar(kXbSFull + i), 1);
      mbar_init(sm.bar(kXbSEmpty + i), kIxEpiWarps);  // every epilogue warp
    }
    for (int i = 0; i < kIxMaxAcc; ++i) {
      mbar_init(sm.bar(kXbTFull + i), 1);
      mbar_init(sm.bar(kXbTEmpty + i), kIxEpiWarps);  // every epilogue warp
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(sm.bar(kXbQFull + i), 1);    // the Q box
      mbar_init(sm.bar(kXbCwFull + i), 32);  // the producer's lanes
      mbar_init(sm.bar(kXbQEmpty + i), 1 + kIxEpiWarps);  // the row's last MMAs and every epilogue warp
    }
    mbar_init(sm.bar(kXbDrain), 1);
    *sm.abort_flag() = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(sm.tmem_slot(), tcols);
  // This CTA's tiles [lo, hi) of all rows' tiles laid end to end: every
  // thread counts the tiles of the rows starting in its run of tokens, a
  // block scan places the runs, and the thread whose run holds tile lo
  // finds the row (and that row's first global tile) it lies in.
  int* scratch = sm.i(kXScan);
  int* plan = sm.plan();
  const int per = (x.T + kIxThreads - 1) / kIxThreads;
  const int t0 = min(x.T, tid * per), t1 = min(x.T, t0 + per);
  int mine = 0;
  for (int t = t0; t < t1; ++t) {
    int b, g;
    mine += ix_row(p, t, x.gmax, x.kcap, b, g);
  }
  int total = 0;
  const int excl = block_exclusive_scan<kIxThreads>(mine, tid, scratch, total);
  const int lo = int((long long)blockIdx.x * total / gridDim.x);
  const int hi = int((long long)(blockIdx.x + 1) * total / gridDim.x);
  if (lo < hi && excl <= lo && lo < excl + mine) {
    int acc = excl;
    for (int t = t0; t < t1; ++t) {
      int b, g;
      const int nt = ix_row(p, t, x.gmax, x.kcap, b, g);
      if (acc + nt > lo) {
        plan[0] = t;
        plan[1] = acc;
        break;
      }
      acc += nt;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_slot();
  if (lo < hi) {
    IxWalk w;
    w.t = plan[0];
    w.start = plan[1];
    w.tiles = ix_row(p, w.t, x.gmax, x.kcap, w.b, w.g);
    if (warp == 0) {
      ix_produce(p, x, sm, w, lo, hi, fault, &kmap, &qmap);
    } else if (warp == 1) {
      if (lane == 0) ix_mma(p, x, sm, w, lo, hi, tmem, fault);
    } else {
      ix_epilogue(p, x, sm, w, lo, hi, tmem, ws, fault);
    }
  }
  if (warp == 1 && lane == 0) {
    // every MMA issued above completes before tensor memory is freed (a
    // bounded wait that an abort does not cut short)
    mma_commit(sm.bar(kXbDrain));
    volatile int never = 0;
    if (!mbar_wait_poll(smem_u32(sm.bar(kXbDrain)), 0, &never, kIxTimeoutNs)) atomicOr(fault, QSFM_FAULT_TIMEOUT);
  }
  // The MMA warp ran on one lane: its lanes meet before the barrier (a
  // barrier reached by part of a warp counts the whole warp).
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
  }
}

// ------------------------------------------------------------- select kernel
constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelBins = 4096;  // 12-bit digits
constexpr int kSelBoundary = 256;  // boundary-bin keys ranked directly (more: further radix passes)
constexpr int kSelCand = 8192;     // keys >= the lower bound listed in shared memory (more: register passes)

// select kernel shared memory: histogram (later the tie bitmap or the
// boundary list), selected-key bitmap, candidate keys and indices, scratch
constexpr size_t kSelSmem = size_t(kSelBins) * 4 + size_t(kIxMaxKeys / 32) * 4 + size_t(kSelCand) * 8 + 128 * 4;

// Exclusive prefix sum over the select's 512 threads with one barrier. The
// warp totals go to half `par` of scr[0..31]; consecutive calls alternate
// halves, so a call never overwrites totals that a warp may still be reading
// from the call before (every warp has passed this call's barrier first).
__device__ __forceinline__ int sel_scan(int v, int tid, int* scr, int par, int& total) {
  const int lane = tid & 31, warp = tid >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  int* tot = scr + 16 * par;
  if (lane == 31) tot[warp] = incl;
  __syncthreads();
  const int wt = lane < kSelWarps ? tot[lane] : 0;
  total = __reduce_add_sync(0xffffffffu, wt);
  return __reduce_add_sync(0xffffffffu, lane < warp ? wt : 0) + incl - v;
}

// One CTA per query token. Thread tid keeps the keys of score groups
// q = tid + 512 i (i < V; four keys 4q .. 4q+3 each) in registers, so a row
// of up to 2048 V scores is read from the workspace once. Absent keys (past
// the row) are 0, below every score's key. The keys at or above a lower
// bound of the k-th largest (about a fifth of a long row) are then listed
// in shared memory, and every later pass runs over that list (over the
// registers when the list would overflow).
template <int V>
__global__ void __launch_bounds__(kSelThreads, V <= 8 ? 2 : 1)
    ix_select_kernel(const qsfm_indexer_params p, const IxShape x, const float* ws, int* fault) {
  extern __shared__ uint4 sel_smem[];
  int* hist = reinterpret_cast<int*>(sel_smem);                  // radix histogram, then tie bitmap / list
  uint32_t* bits = reinterpret_cast<uint32_t*>(hist + kSelBins);  // [kIxMaxKeys / 32] selected keys
  uint32_t* ckey = bits + kIxMaxKeys / 32;                       // [kSelCand] candidate keys
  int* cidx = reinterpret_cast<int*>(ckey + kSelCand);           // [kSelCand] their indices
  int* scratch = cidx + kSelCand;                                // [128]
  uint32_t* uscr = reinterpret_cast<uint32_t*>(scratch);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t = blockIdx.x;
  int b, s, s1, s1e;
  ix_token(p, t, b, s, s1, s1e);
  int nv = s < s1e ? ix_visible(p, b, s, s1) : 0;
  if (nv > x.kcap) {
    if (tid == 0) atomicOr(fault, nv > kIxMaxKeys ? QSFM_FAULT_KV_ROW : QSFM_FAULT_CMP_TABLE_COL);
    nv = x.kcap;
  }
  if (tid == 0 && s == 0 && p.layout_k == QSFM_LAYOUT_KV_TND) {  // a batch past the key tensor (cut in ix_keys)
    const int c0 = __ldg(p.cu_seqlens_k + b), c1 = __ldg(p.cu_seqlens_k + b + 1);
    if (c0 < 0 || c1 > p.total_k) atomicOr(fault, QSFM_FAULT_KV_ROW);
  }
  const int off = p.output_idx_offset != nullptr ? __ldg(p.output_idx_offset + b) : 0;  // added to valid indices
  const int k = p.topk;
  int32_t* out = p.sparse_indices + size_t(t) * k;
  __nv_bfloat16* vals = p.return_value ? static_cast<__nv_bfloat16*>(p.sparse_values) + size_t(t) * k : nullptr;
  const float* sc = ws + size_t(t) * x.kstride;
  grid_dependency_wait();  // the score kernel's rows are complete and visible
  if (nv <= k) {  // every visible key, then -1
    for (int j = tid; j < k; j += kSelThreads) {
      out[j] = j < nv ? j + off : -1;
      if (vals != nullptr) vals[j] = __float2bfloat16_rn(j < nv ? __ldcg(sc + j) : -INFINITY);
    }
    return;
  }
  // 1. The keys, with the smallest, the largest, and this thread's largest.
  // When k is at most the number of threads holding keys, lo = the smallest
  // per-thread largest is a lower bound of the k-th largest key (that many
  // distinct keys are >= lo); otherwise lo is the smallest key.
  const int n4 = (nv + 3) >> 2, nw = (nv + 31) >> 5;
  float4 f[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int q = tid + kSelThreads * i;
    f[i] = q < n4 ? __ldcg(reinterpret_cast<const float4*>(sc) + q) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  uint32_t u[V][4];
  uint32_t kmin = 0xffffffffu, tmax = 0u;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int j = 4 * (tid + kSelThreads * i);
    if (j + 3 < nv) {  // a whole group
      u[i][0] = score_key(f[i].x);
      u[i][1] = score_key(f[i].y);
      u[i][2] = score_key(f[i].z);
      u[i][3] = score_key(f[i].w);
      kmin = min(kmin, min(min(u[i][0], u[i][1]), min(u[i][2], u[i][3])));
    } else {  // the row's last, partial group, or none
      u[i][0] = j < nv ? score_key(f[i].x) : 0u;
      u[i][1] = j + 1 < nv ? score_key(f[i].y) : 0u;
      u[i][2] = j + 2 < nv ? score_key(f[i].z) : 0u;
      u[i][3] = j + 3 < nv ? score_key(f[i].w) : 0u;
      if (j < nv) kmin = min(kmin, u[i][0]);
      if (j + 1 < nv) kmin = min(kmin, u[i][1]);
      if (j + 2 < nv) kmin = min(kmin, u[i][2]);
    }
    tmax = max(tmax, max(max(u[i][0], u[i][1]), max(u[i][2], u[i][3])));
  }
  for (int i = tid; i < nw; i += kSelThreads) bits[i] = 0u;
  if (tid == 0) scratch[99] = 0;  // candidate count
  int sp = 0;                     // scan parity (sel_scan)
  {
    const uint32_t a = __reduce_min_sync(0xffffffffu, kmin);
    const uint32_t c = __reduce_max_sync(0xffffffffu, tmax);
    const uint32_t o = __reduce_min_sync(0xffffffffu, tid < n4 ? tmax : 0xffffffffu);
    if (lane == 0) {
      uscr[warp] = a;
      uscr[kSelWarps + warp] = c;
      uscr[2 * kSelWarps + warp] = o;
    }
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t a = lane < kSelWarps ? uscr[lane] : 0xffffffffu;
    uint32_t c = lane < kSelWarps ? uscr[kSelWarps + lane] : 0u;
    uint32_t o = lane < kSelWarps ? uscr[2 * kSelWarps + lane] : 0xffffffffu;
    a = __reduce_min_sync(0xffffffffu, a);
    c = __reduce_max_sync(0xffffffffu, c);
    o = __reduce_min_sync(0xffffffffu, o);
    if (lane == 0) {
      uscr[100] = a;
      uscr[101] = c;
      uscr[102] = o;
    }
  }
  __syncthreads();
  const uint32_t kmax = uscr[101];
  const uint32_t lo = k <= min(kSelThreads, n4) ? uscr[102] : uscr[100];

  // 2. The candidates (keys >= lo, among them the k-th largest), listed in
  // any order: each warp takes one slot range (a warp scan and one shared
  // atomic); what does not fit is not written, and then the later passes
  // run over the registers.
  int mine = 0;
#pragma unroll
  for (int i = 0; i < V; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) mine += u[i][e] >= lo;
  {
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int base = 0;
    if (lane == 31 && incl > 0) base = atomicAdd(&scratch[99], incl);
    int off = __shfl_sync(0xffffffffu, base, 31) + incl - mine;
#pragma unroll
    for (int i = 0; i < V; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (u[i][e] >= lo) {
          if (off < kSelCand) {
            ckey[off] = u[i][e];
            cidx[off] = 4 * (tid + kSelThreads * i) + e;
          }
          ++off;
        }
  }
  __syncthreads();
  const int ncand = scratch[99];
  const bool listed = ncand <= kSelCand;

  // 3. Radix select of the k-th largest candidate. The candidates share the
  // bits of lo and kmax above the highest bit where those two differ; the
  // digits (12 bits at most) start below. A candidate is taken when its bits
  // under `mask` beat `prefix`, or equal it and it is among the first `need`
  // such (by score, then key index); `eq` counts those equal to the prefix.
  // Passes stop once the boundary bin is taken whole or holds few enough
  // candidates to rank directly.
  uint32_t mask, prefix;
  int need, eq = -1;  // -1: not counted
  const uint32_t diff = lo ^ kmax;
  if (diff == 0u) {  // every candidate is equal: the first k of them
    mask = 0xffffffffu;
    prefix = kmax;
    need = k;
  } else {
    int nbits = 32 - __clz(diff);
    mask = nbits == 32 ? 0u : ~((1u << nbits) - 1u);
    prefix = kmax & mask;
    int remaining = k;  // of the candidates matching the prefix, the rank wanted
    while (nbits > 0) {
      const int d = min(12, nbits), shift = nbits - d, nb = 1 << d;
      for (int i = tid; i < nb; i += kSelThreads) hist[i] = 0;
      __syncthreads();
      if (listed) {
        for (int c = tid; c < ncand; c += kSelThreads) {
          const uint32_t v = ckey[c];
          if ((v & mask) == prefix) atomicAdd(&hist[(v >> shift) & uint32_t(nb - 1)], 1);
        }
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t v = u[i][e];
            if (v >= lo && (v & mask) == prefix) atomicAdd(&hist[(v >> shift) & uint32_t(nb - 1)], 1);
          }
      }
      __syncthreads();
      // thread i sums bins nb-1-i*per down to nb-i*per-per (largest first)
      const int per = (nb + kSelThreads - 1) / kSelThreads;
      const int top = nb - 1 - tid * per;
      int sum = 0;
      for (int q = 0; q < per; ++q)
        if (top - q >= 0) sum += hist[top - q];
      int tot = 0;
      const int ex = sel_scan(sum, tid, scratch, sp, tot);
      sp ^= 1;
      if (ex < remaining && remaining <= ex + sum) {  // exactly one thread
        int acc = ex;
        for (int q = 0; q < per; ++q) {
          const int c = hist[top - q];
          if (acc + c >= remaining) {
            scratch[96] = top - q;
            scratch[97] = acc;  // candidates in larger bins
            scratch[98] = c;
            break;
          }
          acc += c;
        }
      }
      __syncthreads();
      prefix |= uint32_t(scratch[96]) << shift;
      mask |= uint32_t(nb - 1) << shift;
      remaining -= scratch[97];
      eq = scratch[98];
      nbits = shift;
      __syncthreads();
      if (eq == remaining || eq <= kSelBoundary) break;  // taken whole, or ranked below
    }
    need = remaining;
  }

  // 4. Mark the selected keys: every candidate above the prefix; the equal
  // ones too when all of them are taken. Otherwise a few equal ones are
  // listed and ranked (score, then key index) directly; many (ties past the
  // k-th) go through a tie bitmap in key order.
  const bool all_eq = eq == need;
  const bool few = !all_eq && eq >= 0 && eq <= kSelBoundary;
  uint32_t* tbits = reinterpret_cast<uint32_t*>(hist);  // kcap / 32 <= 1024 words
  uint32_t* lkey = reinterpret_cast<uint32_t*>(hist);   // boundary keys [256]
  int* lidx = hist + kSelBoundary;                      // and their indices [256]
  if (!all_eq && !few)
    for (int i = tid; i < nw; i += kSelThreads) tbits[i] = 0u;
  if (tid == 0) scratch[95] = 0;  // boundary count (scratch[99] still holds the candidate count)
  __syncthreads();
  auto mark = [&](uint32_t v, int j) {
    const uint32_t hv = v & mask;
    if (hv > prefix || (hv == prefix && all_eq)) {
      atomicOr(&bits[j >> 5], 1u << (j & 31));
    } else if (hv == prefix) {
      if (few) {
        const int slot = atomicAdd(&scratch[95], 1);  // < eq <= 256
        lkey[slot] = v;
        lidx[slot] = j;
      } else {
        atomicOr(&tbits[j >> 5], 1u << (j & 31));
      }
    }
  };
  if (listed) {
    for (int c = tid; c < ncand; c += kSelThreads) mark(ckey[c], cidx[c]);
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (u[i][e] >= lo) mark(u[i][e], 4 * (tid + kSelThreads * i) + e);
  }
  __syncthreads();
  if (few) {  // warp w ranks boundary keys w, w + 16, ...: larger first, then smaller index
    for (int c = warp; c < eq; c += kSelWarps) {
      const uint32_t v = lkey[c];
      const int j = lidx[c];
      int rank = 0;
      for (int o = lane; o < eq; o += 32) {
        const uint32_t w2 = lkey[o];
        rank += w2 > v || (w2 == v && lidx[o] < j);
      }
      rank = __reduce_add_sync(0xffffffffu, rank);
      if (lane == 0 && rank < need) atomicOr(&bits[j >> 5], 1u << (j & 31));
    }
    __syncthreads();
  } else if (!all_eq) {  // thread i owns tie words 2i, 2i + 1 (nw <= 1024)
    const int w0 = 2 * tid;
    const uint32_t t0 = w0 < nw ? tbits[w0] : 0u, t1 = w0 + 1 < nw ? tbits[w0 + 1] : 0u;
    int tot = 0;
    int r = sel_scan(__popc(t0) + __popc(t1), tid, scratch, sp, tot);
    sp ^= 1;
    const uint32_t m[2] = {t0, t1};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t take = 0u;
      for (uint32_t v = m[h]; v != 0u && r < need; v &= v - 1u, ++r) take |= v & (~v + 1u);
      if (take != 0u) bits[w0 + h] |= take;  // the words are this thread's alone
    }
    __syncthreads();
  }

  // 5. The marked keys in ascending order: thread i owns words 2i, 2i + 1.
  const int w0 = 2 * tid;
  const uint32_t b0 = w0 < nw ? bits[w0] : 0u, b1 = w0 + 1 < nw ? bits[w0 + 1] : 0u;
  int tot = 0;
  int pos = sel_scan(__popc(b0) + __popc(b1), tid, scratch, sp, tot);
  const uint32_t m[2] = {b0, b1};
#pragma unroll
  for (int h = 0; h < 2; ++h)
    for (uint32_t v = m[h]; v != 0u; v &= v - 1u, ++pos) {
      const int j = 32 * (w0 + h) + (__ffs(v) - 1);
      out[pos] = j + off;
      if (vals != nullptr) vals[pos] = __float2bfloat16_rn(__ldcg(sc + j));
    }
}

template <int V>
cudaError_t launch_select(const qsfm_indexer_params& p, const IxShape& x, const float* ws, int* fault,
                          cudaStream_t s) {
  const cudaError_t e =
      cudaFuncSetAttribute(ix_select_kernel<V>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSelSmem));
  if (e != cudaSuccess) return e;
  return launch_after_predecessor(ix_select_kernel<V>, dim3(x.T), dim3(kSelThreads), kSelSmem, s, p, x, ws,
                                  fault);
}

// ------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult qres;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qres) ==
            cudaSuccess &&
        qres == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return encode;
}

// The keys viewed as [rows, 128 bytes] (the paged pool's num_blocks * 128
// rows, the BSND slabs' B * S_k, the TND tensor's T_k), boxes of 128 rows x
// 128 bytes with the 128-byte swizzle of the MMA's K-major operand.
cudaError_t make_key_map(const void* key, long long rows, CUtensorMap* map) {
  const auto encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cuuint64_t(kIxDim), cuuint64_t(rows > 0 ? rows : 1)};
  const cuuint64_t strides[1] = {cuuint64_t(kIxDim)};
  const cuuint32_t box[2] = {kIxDim, kIxTile};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(key), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The queries viewed as [T, heads, 128 bytes]; a box is one row of the score
// kernel: gmax tokens x hp heads (heads past the real ones, and tokens past
// T, read as zero), laid out as gmax * hp rows of 128 bytes with the 128-byte
// swizzle, the MMA's K-major B operand.
cudaError_t make_query_map(const void* query, int heads, int T, int hp, int gmax, CUtensorMap* map) {
  const auto encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {cuuint64_t(kIxDim), cuuint64_t(heads), cuuint64_t(T)};
  const cuuint64_t strides[2] = {cuuint64_t(kIxDim), cuuint64_t(heads) * kIxDim};
  const cuuint32_t box[3] = {kIxDim, cuuint32_t(hp), cuuint32_t(gmax)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(query), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

IxShape indexer_shape(const qsfm_indexer_params& p, int T) {
  IxShape x;
  x.T = T;
  x.hp = (p.heads + 15) & ~15;
  x.gmax = kIxMaxN / x.hp < kIxMaxG ? kIxMaxN / x.hp : kIxMaxG;
  if (p.layout_q == QSFM_LAYOUT_BSND && p.max_s1 < x.gmax) x.gmax = p.max_s1;
  x.paged = p.layout_k == QSFM_LAYOUT_KV_PA_BBND;
  const long long keys = x.paged ? (long long)p.max_blocks * kIxTile
                                 : p.layout_k == QSFM_LAYOUT_KV_BSND ? (long long)p.max_sk : (long long)p.total_k;
  x.kcap = int(keys < kIxMaxKeys ? keys : kIxMaxKeys);
  x.kstride = x.kcap < kIxTile ? kIxTile : (x.kcap + kIxTile - 1) & ~(kIxTile - 1);  // whole tiles of scores
  x.nacc = (x.gmax * x.hp + 31) & ~31;
  x.na = kIxMaxAcc * x.nacc <= 512 ? kIxMaxAcc : 2;
  x.tcols = 32;
  while (x.tcols < x.na * x.nacc) x.tcols <<= 1;
  x.qslot = (x.gmax * x.hp * kIxDim + 1023) & ~1023;
  const int room = int(kXSmemMax) - 1024 - int(kXFixed) - 2 * x.qslot;
  x.stages = room / int(kXStage) < kIxMaxStages ? room / int(kXStage) : kIxMaxStages;
  return x;
}

}  // namespace

size_t indexer_workspace_bytes(const qsfm_indexer_params& p, int num_tokens) {
  return size_t(num_tokens) * size_t(indexer_shape(p, num_tokens).kstride) * sizeof(float);
}

cudaError_t launch_indexer(const qsfm_indexer_params& p, int T, void* workspace, int* fault, cudaStream_t s) {
  const IxShape x = indexer_shape(p, T);
  cudaError_t e =
      cudaFuncSetAttribute(ix_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(x.smem_bytes()));
  if (e != cudaSuccess) return e;
  CUtensorMap kmap, qmap;
  const long long key_rows = x.paged ? (long long)p.num_blocks * kIxTile
                             : p.layout_k == QSFM_LAYOUT_KV_BSND ? (long long)p.batch * p.max_sk : (long long)p.total_k;
  if ((e = make_key_map(p.key, key_rows, &kmap)) != cudaSuccess) return e;
  if ((e = make_query_map(p.query, p.heads, T, x.hp, x.gmax, &qmap)) != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  float* ws = static_cast<float*>(workspace);
  ix_score_kernel<<<sms, kIxThreads, x.smem_bytes(), s>>>(p, x, ws, fault, kmap, qmap);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // keys per thread: the row's 4-score groups over 512 threads, rounded up
  // to a power of two
  const int v = (x.kcap + 4 * kSelThreads - 1) / (4 * kSelThreads);
  const float* cws = ws;
  if (v <= 1) return launch_select<1>(p, x, cws, fault, s);
  if (v <= 2) return launch_select<2>(p, x, cws, fault, s);
  if (v <= 4) return launch_select<4>(p, x, cws, fault, s);
  if (v <= 8) return launch_select<8>(p, x, cws, fault, s);
  return launch_select<16>(p, x, cws, fault, s);
}

}  // namespace qsfm
