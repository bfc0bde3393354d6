// Attention kernel of the quantized shared-KV sparse MLA forward (sm_103a).
//
// Computes, for every planned (work unit, KV-tile range) piece,
//   O = softmax([Q K~^T * softmax_scale, sink]) V~  with K~ = V~
// (QuantSparseFlashMla, function description formula; sink from its
// parameter table row "sinks"; lse from KvQuantSparseAttnSharedKv, parameter
// table row softmax_lse).
//
// Orientation. The contractions run transposed so that the KV rows of a tile
// (128 rows) are the M dimension of the score product and the 64 heads of a
// unit are N:
//   S^T[j, h]  = sum_d K~[j, d] Q[h, d]      (M = 128 rows, N = 64, K = 512)
//   O^T[d, h] += sum_j V~[j, d] P[h, j]      (M = 128 d per chunk, N = 64,
//                                             K = 128 rows, 4 chunks)
// Both accumulators live in tensor memory: S^T in 64 columns (lane = tile
// row), O^T in 256 columns (lane = head-dim element of a 128-wide chunk).
// The dequantised bf16 tile (128 rows x 512, eight 16 KB slabs of 64 d with
// the 128-byte swizzle) is the K-major A operand of the first product and,
// read through an MN-major descriptor, the A operand of the second: each row
// is dequantised once and read by both products.
//
// Pipeline. One tile buffer, in four chunks of two slabs (128 d each). The
// single MMA-issuing thread runs, per tile n:
//   PV(n) chunks 0..3 (a commit after chunks 1 and 3 frees them in pairs),
//   then QK^T(n + 1) chunks 0..3 as the workers refill them with tile n + 1,
// so the workers store chunks 0 and 1 of tile n + 1 while the tensor cores
// run chunks 2 and 3 of PV(n). Only the softmax of a tile (between its last
// QK^T MMA and its first PV MMA) leaves the tensor pipe idle. Commits are
// kept few: each one drains the tensor pipe (about 140 cycles).
//
// Warp roles (10 warps, at most 3 per SM sub-partition, so up to 168
// registers per thread):
//   warps 0-7   workers: each tile's softmax, the production of the next
//               tile and each unit's epilogue, in that order.
//               Softmax / epilogue view: warp w reads tensor-memory lanes
//               32 (w % 4) .. + 31 (tile rows, or head-dim elements of a
//               128-wide O^T chunk) and heads 32 (w / 4) .. + 31; each thread
//               writes its P values (bf16, the MN-major B operand of PV);
//               lane i keeps the running sum of P for head 32 (w / 4) + i
//               over the warp's rows.
//               Producer view: thread (row_lo, j) holds rows row_lo + 32 u
//               (u < 4) of the next tile, raw, in registers (all four
//               chunks for fp8 and packed rows; two for bf16 rows); once PV
//               has read a chunk's slabs it dequantises that chunk (fp8 ->
//               f16 -> fp32 x scale -> bf16), stores and publishes it; after
//               the last chunk it loads the tile after next, which then has
//               a whole tile's time in flight.
//   warp 8      MMA issue (one thread): Q by TMA, PV and QK^T as above.
//   warp 9      resolver: turns the tiles' slots into physical rows (sparse
//               indices, block tables, masks), four tiles per pass with all
//               their loads in flight together, up to 8 tiles ahead, into a
//               shared-memory ring, and asks L2 for each new unit's Q.
// mbarriers carry every hand-off; every wait is bounded in time.
//
// Softmax: the running max m_used per head is moved only when a tile's max
// exceeds it by more than 8 (log2 units); a named-barrier vote detects that
// case, so most tiles need no cross-row max reduction. When it moves, O^T
// and the row sums are rescaled exactly. P <= 2^8 in bf16.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "qsfm_device.cuh"
#include "qsfm_internal.h"

namespace qsfm {
namespace {

static_assert(kTileRows == 128, "the kernel's layouts assume 128-row tiles");

constexpr int kWorkWarps = 8;
constexpr int kWorkThreads = kWorkWarps * 32;
constexpr int kHPT = 256 / kWorkWarps;       // heads per worker thread (softmax, epilogue)
constexpr int kRPT = 32 / kWorkWarps;        // tile rows per worker thread (producer)
constexpr int kRowStride = 4 * kWorkWarps;   // between a producer thread's rows
static_assert(kHPT == 16 || kHPT == 32, "worker warps: 8 or 16");
constexpr int kMmaWarp = kWorkWarps;
constexpr int kResolverWarp = kMmaWarp + 1;
constexpr int kThreads = (kResolverWarp + 1) * 32;
constexpr int kRing = 8;     // tiles of resolved rows in flight
constexpr int kResolveTiles = 1;  // tiles per resolver pass (more keeps more loads in flight, at a
                                  // larger instruction footprint; the ring already runs 8 tiles ahead)
constexpr int kBarWork = 1;  // named barrier id of the worker warps

// shared memory map (byte offsets from a 1024-aligned base)
constexpr uint32_t kSlabBytes = kTileRows * 128;                // 128 rows x 64 d (bf16): 16 KB
constexpr uint32_t kSK = 0;                                     // K~ tile: 8 slabs
constexpr uint32_t kSQ = kSK + 8 * kSlabBytes;                  // Q: 8 d-blocks x 64 heads x 128 B
constexpr uint32_t kSP = kSQ + 8 * 64 * 128;                    // P: 128 rows x 64 heads (bf16)
constexpr uint32_t kSRows = kSP + kTileRows * 128;              // [kRing][128] i32 physical rows
constexpr uint32_t kSRowKind = kSRows + kRing * kTileRows * 4;  // [kRing] i32: 0 ori, 1 cmp, -1 end
constexpr uint32_t kSValid = kSRowKind + 64;                    // [128] i32: row of the tile valid
constexpr uint32_t kSRed = kSValid + kTileRows * 4;             // [4][64] f32 per-quadrant partials
constexpr uint32_t kSMUsed = kSRed + 1024;                      // [64] f32
constexpr uint32_t kSAlpha = kSMUsed + 256;                     // [64] f32
constexpr uint32_t kSInv = kSAlpha + 256;                       // [64] f32
constexpr uint32_t kSBar = kSInv + 256;                         // mbarriers, tmem base, flags
constexpr uint32_t kSmemBytes = kSBar + 256;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
static_assert(kSmemAlloc <= 232448, "more than the 227 KB a CTA may use");

// mbarrier slots
constexpr int kBarQFull = 0;
constexpr int kBarFull = 1;       // [chunk]: stored (one arrive per worker warp)
constexpr int kBarFree = 5;       // [chunk pair]: PV of chunks 2i, 2i + 1 completed (commit)
constexpr int kBarSFull = 7;      // S^T of the tile complete (commit)
constexpr int kBarPFull = 8;      // P of the tile written (one arrive per worker warp)
constexpr int kBarOFree = 9;      // O^T read by the epilogue (one arrive per worker warp)
constexpr int kBarDrain = 10;     // every MMA of the CTA completed (commit)
constexpr int kBarQReady = 27;    // Q converted to f16 (one arrive per worker warp; fp8 rows)
constexpr int kBarRowsFull = 11;  // [ring slot]
constexpr int kBarRowsEmpty = 19; // [ring slot], one arrive per worker warp
constexpr int kNumBars = 28;
static_assert(kNumBars * 8 <= 224, "barriers overlap the tmem slot");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = 256;  // + 64 * chunk
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Operand type of the products: fp8 rows are dequantised to f16 (one exact
// e4m3 -> f16 conversion and one f16 multiply per pair of values; q is
// converted to f16 when it lands, with an exact power-of-two prescale);
// packed and bf16 rows keep bf16 (their bf16 rope / rows need its range).
template <int kFmt>
constexpr bool kF16Ops = kFmt == QSFM_KV_FP8_FP32_SCALES;
template <int kFmt>
constexpr uint32_t kIdescQK = make_idesc_bf16(128, 64, /*a_mn=*/0, /*b_mn=*/0, kF16Ops<kFmt>);
template <int kFmt>
constexpr uint32_t kIdescPV = make_idesc_bf16(128, 64, /*a_mn=*/1, /*b_mn=*/1, kF16Ops<kFmt>);
// Largest per-row power-of-two prescale of fp8 rows: P (<= 2^8 by the lazy
// max) times 2^7 stays inside f16.
constexpr int kMaxRowShift = 7;
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait

struct Range {
  int t0, k0, t1, k1;
};

// Walks the (unit, tile-range) pieces of a CTA's range in order.
struct PieceIter {
  const qsfm_params* p;
  Range r;
  int T;
  int t;
  __device__ PieceIter(const qsfm_params* p_, Range r_, int T_) : p(p_), r(r_), T(T_), t(r_.t0) {}
  __device__ bool next(int& tok, TokenGeom& g, int& lo, int& hi) {
    if (t > r.t1 || t >= T || (t == r.t1 && r.k1 == 0)) return false;
    tok = t;
    g = token_geom(*p, t);
    lo = (t == r.t0) ? min(r.k0, g.n_tiles) : 0;
    hi = (t == r.t1) ? min(r.k1, g.n_tiles) : g.n_tiles;
    ++t;
    return true;
  }
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Max (kMax) or sum of kN (16 or 32) values per lane over the 32 lanes of a
// warp, by halving exchanges (for kN = 16, lanes l and l ^ 16 are combined
// first): afterwards lane l holds the result for value index l % kN. The
// array is consumed.
template <bool kMax, int kN>
__device__ __forceinline__ float reduce_lanes(float (&v)[kN]) {
  const int lane = threadIdx.x & 31;
  if constexpr (kN == 16) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float got = __shfl_xor_sync(0xffffffffu, v[i], 16);
      v[i] = kMax ? fmaxf(v[i], got) : v[i] + got;
    }
  }
#pragma unroll
  for (int w = kN / 2; w >= 1; w >>= 1) {
    const bool up = lane & w;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float keep = up ? v[w + i] : v[i];
      const float send = up ? v[i] : v[w + i];
      const float got = __shfl_xor_sync(0xffffffffu, send, w);
      v[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
  return v[0];
}

// kN consecutive tensor-memory columns of the warp's 32 lanes, one lane per
// thread.
template <int kN>
__device__ __forceinline__ void tmem_load(uint32_t taddr, float (&v)[kN]) {
  if constexpr (kN == 32) tmem_ld32(taddr, v);
  else tmem_ld16(taddr, v);
}
template <int kN>
__device__ __forceinline__ void tmem_store(uint32_t taddr, const float (&v)[kN]) {
  if constexpr (kN == 32) tmem_st32(taddr, v);
  else tmem_st16(taddr, v);
}

struct Smem {
  uint32_t base;
  uint8_t* ptr;
  __device__ float* f(uint32_t off) const { return reinterpret_cast<float*>(ptr + off); }
  __device__ uint64_t* bar(int i) const { return reinterpret_cast<uint64_t*>(ptr + kSBar) + i; }
  __device__ uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(ptr + kSBar + 224); }
  __device__ volatile int* abort_flag() const {
    return reinterpret_cast<volatile int*>(ptr + kSBar + 232);
  }
};

// Bounded wait; on timeout raises the CTA's abort flag and the fault bit.
__device__ __forceinline__ bool wait_or_abort(const Smem& sm, int bar, uint32_t parity, int* fault) {
  if (mbar_wait_bounded(sm.bar(bar), parity, sm.abort_flag(), kTimeoutNs)) return true;
  if (!*sm.abort_flag()) {
    *sm.abort_flag() = 1;
    atomicOr(fault, QSFM_FAULT_TIMEOUT);
  }
  return false;
}

// Warp-uniform bounded wait: lane 0 polls, the result is broadcast, so the
// lanes of a warp never split on a timeout.
__device__ __forceinline__ bool warp_wait_or_abort(const Smem& sm, int bar, uint32_t parity,
                                                   int* fault) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = wait_or_abort(sm, bar, parity, fault);
  __syncwarp();  // the other lanes wait here (and are ordered after lane 0's acquire)
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// Asks L2 for the bytes of physical row `prow` of a pool (and its scale row).
template <int kFmt>
__device__ __forceinline__ void prefetch_row(const uint8_t* pool, const float* spool, int prow) {
  constexpr uint32_t kRowB = kv_row_bytes(kFmt);
  bulk_prefetch_l2(pool + size_t(prow) * kRowB, kRowB);
  if constexpr (kFmt == QSFM_KV_FP8_FP32_SCALES) prefetch_l2(spool + size_t(prow) * kScales);
}

// ------------------------------------------------------------- resolver
// Tile n's rows go to ring slot n % kRing: 128 physical rows (block * 128 +
// offset, -1 = masked) and the pool they come from. After the CTA's last tile
// the resolver writes an end mark (-1) in the next slot. Up to kResolveTiles
// tiles of one unit per pass: all their index loads are in flight together,
// then all their block-table loads, so a pass costs two memory round trips
// whatever its tile count.
template <int kFmt>
__device__ void resolver_role(const qsfm_params& p, const Smem& sm, Range rg, int T, int* fault) {
  constexpr int kN = kResolveTiles;
  const int lane = threadIdx.x & 31;
  int* rows = reinterpret_cast<int*>(sm.ptr + kSRows);
  int* kind = reinterpret_cast<int*>(sm.ptr + kSRowKind);
  const uint8_t* q8 = static_cast<const uint8_t*>(p.q);
  PieceIter pieces(&p, rg, T);
  uint32_t n = 0;  // next ring position
  int unit, lo, hi;
  TokenGeom g;
  while (pieces.next(unit, g, lo, hi)) {
    if (lo >= hi) continue;
    // the unit's Q goes to L2 a few tiles before its first product; the next
    // token's index list while this one is resolved
    if (lane == 0) bulk_prefetch_l2(q8 + size_t(unit) * kHeads * kDim * 2, kHeads * kDim * 2);
    if (p.cmp_sparse_indices != nullptr && g.tok + 1 < (T >> unit_shift(p))) {
      const uint8_t* ix = reinterpret_cast<const uint8_t*>(p.cmp_sparse_indices + (size_t)(g.tok + 1) * p.k2);
      for (int off = 128 * lane; off < 4 * p.k2; off += 32 * 128) prefetch_l2(ix + off);
    }
    // passes of up to kN tiles of this unit
    for (int k0 = lo; k0 < hi; k0 += kN) {
      int k[kN];
      bool live[kN];
#pragma unroll
      for (int t = 0; t < kN; ++t) {
        k[t] = k0 + t;
        live[t] = k0 + t < hi;
      }
#pragma unroll
      for (int t = 0; t < kN; ++t) {
        const uint32_t m = n + t;
        if (live[t] && !warp_wait_or_abort(sm, kBarRowsEmpty + m % kRing, ((m / kRing) & 1) ^ 1, fault)) return;
      }
      int lg[kN][4], pr[kN][4];
      bool cmp[kN];
      resolve_tile_rows<kN>(p, g, k, live, lane, fault, lg, pr, cmp);
#pragma unroll
      for (int t = 0; t < kN; ++t) {
        if (!live[t]) continue;
        const uint32_t slot = (n + t) % kRing;
#pragma unroll
        for (int u = 0; u < 4; ++u) rows[slot * kTileRows + lane + 32 * u] = pr[t][u];
        if (lane == 0) kind[slot] = cmp[t] ? 1 : 0;
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.bar(kBarRowsFull + slot));
      }
      n += min(kN, hi - k0);
    }
  }
  // end mark after the CTA's last tile
  const uint32_t slot = n % kRing;
  if (!warp_wait_or_abort(sm, kBarRowsEmpty + slot, ((n / kRing) & 1) ^ 1, fault)) return;
  if (lane == 0) kind[slot] = -1;
  __syncwarp();
  if (lane == 0) mbar_arrive(sm.bar(kBarRowsFull + slot));
}

__device__ __forceinline__ float e8m0_value(uint32_t e) {
  // 2^(e - 127): the fp32 with biased exponent e (e = 0: the subnormal 2^-127)
  return e == 0xFFu ? __uint_as_float(0x7FC00000u) : e == 0u ? __uint_as_float(0x00400000u)
                                                             : __uint_as_float(e << 23);
}

// ------------------------------------------------------------- MMA issue
// QK^T of chunk c (d-blocks 2c, 2c + 1), k-step s of d-block db: A (K~,
// K-major) at + db * 16 KB + s * 32 B, B (Q, K-major) at + db * 8 KB + s * 32
// B. The chunk is a runtime argument (one copy of the code for all four);
// its eight MMAs are unrolled with constant offsets from the chunk's base
// descriptors, so the issuing thread keeps ahead of the tensor pipe.
template <int kFmt, uint32_t kDb, uint32_t kS>
__device__ __forceinline__ void qk_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
  mma_f16_at<((kDb * kSlabBytes + kS * 32) >> 4), ((kDb * 8192 + kS * 32) >> 4)>(d, a, b, kIdescQK<kFmt>, acc);
}

template <int kFmt>
__device__ __forceinline__ void qk_chunk(uint32_t d, uint64_t a0, uint64_t b0, int c) {
  const uint64_t a = a0 + ((uint32_t(c) * 2 * kSlabBytes) >> 4);
  const uint64_t b = b0 + ((uint32_t(c) * 2 * 8192) >> 4);
  qk_mma<kFmt, 0, 0>(d, a, b, c != 0 ? 1u : 0u);
  qk_mma<kFmt, 0, 1>(d, a, b, 1u); qk_mma<kFmt, 0, 2>(d, a, b, 1u); qk_mma<kFmt, 0, 3>(d, a, b, 1u);
  qk_mma<kFmt, 1, 0>(d, a, b, 1u); qk_mma<kFmt, 1, 1>(d, a, b, 1u);
  qk_mma<kFmt, 1, 2>(d, a, b, 1u); qk_mma<kFmt, 1, 3>(d, a, b, 1u);
}

// PV of head-dim chunk c, k-step s: A (V~^T, MN-major: 64-d atoms 16 KB
// apart, 8-row groups 1 KB apart) at + c * 32 KB + s * 2 KB, B (P^T,
// MN-major) at + s * 2 KB; accumulates into O^T columns 64 c .. + 63.
template <int kFmt, uint32_t kS>
__device__ __forceinline__ void pv_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
  mma_f16_at<((kS * 2048) >> 4), ((kS * 2048) >> 4)>(d, a, b, kIdescPV<kFmt>, acc);
}

template <int kFmt>
__device__ __forceinline__ void pv_chunk(uint32_t tmem, uint64_t a0, uint64_t b0, uint32_t acc0, int c) {
  const uint32_t d = tmem + kTmemO + uint32_t(c) * 64;
  const uint64_t a = a0 + ((uint32_t(c) * 2 * kSlabBytes) >> 4);
  pv_mma<kFmt, 0>(d, a, b0, acc0);
  pv_mma<kFmt, 1>(d, a, b0, 1u); pv_mma<kFmt, 2>(d, a, b0, 1u); pv_mma<kFmt, 3>(d, a, b0, 1u);
  pv_mma<kFmt, 4>(d, a, b0, 1u); pv_mma<kFmt, 5>(d, a, b0, 1u);
  pv_mma<kFmt, 6>(d, a, b0, 1u); pv_mma<kFmt, 7>(d, a, b0, 1u);
}

// Tile n of the CTA's sequence: every per-tile barrier completes once per
// tile, so a wait for tile n uses phase parity n & 1. A phase can never run
// two ahead of its waiter: each completion needs the waiter's own next step.
template <int kFmt>
__device__ void mma_role(const qsfm_params& p, const Smem& sm, Range rg, int T, uint32_t tmem,
                         const CUtensorMap* qmap, int* fault) {
  // Q of a piece is ready for its products once it has landed (bf16 rows)
  // or once the workers have converted it to f16 (fp8 rows)
  constexpr int kBarQ = kF16Ops<kFmt> ? kBarQReady : kBarQFull;
  if ((threadIdx.x & 31) != 0) return;
  PieceIter pieces(&p, rg, T);
  TokenGeom g;
  auto next_live = [&](int& t_, int& lo_, int& hi_) {
    while (pieces.next(t_, g, lo_, hi_))
      if (lo_ < hi_) return true;
    return false;
  };
  auto load_q = [&](int unit) {
    mbar_arrive_expect_tx(sm.bar(kBarQFull), kHeads * kDim * 2);
#pragma unroll
    for (int db = 0; db < 8; ++db)
      tma_load_2d(sm.base + kSQ + db * 8192, qmap, db * 64, unit * 64, sm.bar(kBarQFull));
  };
  const uint64_t qa = make_sdesc_sw128(sm.base + kSK, 16, 1024);
  const uint64_t qb = make_sdesc_sw128(sm.base + kSQ, 16, 1024);
  const uint64_t pa = make_sdesc_sw128(sm.base + kSK, kSlabBytes, 1024);
  const uint64_t pb = make_sdesc_sw128(sm.base + kSP, 16, 1024);
  const uint32_t ds = tmem + kTmemS;
  // QK^T of tile n, chunk by chunk as the producers publish the chunks
  auto qk_tile = [&](uint32_t n) -> bool {
    const uint32_t par = n & 1;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      if (!wait_or_abort(sm, kBarFull + c, par, fault)) return false;
      tc_fence_after();
      qk_chunk<kFmt>(ds, qa, qb, c);
    }
    mma_commit(sm.bar(kBarSFull));
    return true;
  };

  int tok, lo, hi;
  if (!next_live(tok, lo, hi)) return;
  load_q(tok);
  uint32_t n = 0, piece = 0;
  bool have = true;
  while (have) {
    int ntok = 0, nlo = 0, nhi = 0;
    const bool have_next = next_live(ntok, nlo, nhi);
#pragma unroll 1
    for (int k = lo; k < hi; ++k, ++n) {
      const bool last = k == hi - 1;
      // QK^T(n) right after PV(n - 1): the piece's q first
      if (k == lo && !wait_or_abort(sm, kBarQ, piece & 1, fault)) return;
      if (!qk_tile(n)) return;
      // P(n) written (so S^T(n) has been read and QK^T(n) is complete)
      if (!wait_or_abort(sm, kBarPFull, n & 1, fault)) return;
      tc_fence_after();
      if (k == lo && piece > 0) {
        // the previous piece's epilogue must have read O^T before it is overwritten
        if (!wait_or_abort(sm, kBarOFree, (piece - 1) & 1, fault)) return;
        tc_fence_after();
      }
      if (last && have_next) load_q(ntok);  // Q is free: QK^T(n) has completed
      // Two commits per tile (each drains the tensor pipe for about 140
      // cycles): chunks 0 and 1 are freed first, so the producers store the
      // next tile's chunks 0 and 1 while chunks 2 and 3 are multiplied.
      const uint32_t acc0 = k == lo ? 0u : 1u;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        pv_chunk<kFmt>(tmem, pa, pb, acc0, c);
        if (c & 1) mma_commit(sm.bar(kBarFree + (c >> 1)));
      }
    }
    ++piece;
    have = have_next;
    tok = ntok;
    lo = nlo;
    hi = nhi;
  }
}

// ------------------------------------------------------------- workers
// Producer view, thread (row_lo, j): rows row_lo + kRowStride u (u < kRPT)
// of a tile, 16-byte piece j of each 128-d chunk c (d 128 c .. 128 c + 127):
//   fp8 rows     fp8 bytes 128 c + 16 j .. + 15 of the row (d 128 c + 16 j
//                .. + 15, d-block 2 c + j / 4, scale index 2 c + j / 4; lane
//                j holds scale j of each of its rows);
//   packed rows  chunk 0: bf16 rope bytes 16 j .. + 15 (d 8 j .. + 7 of
//                d-block 0) and, for j < 4, nope bytes 128 + 16 j .. + 15
//                (d 64 + 16 j .., d-block 1, e8m0 scale 0); chunk c >= 1:
//                nope bytes 64 + 128 c + 16 j .. + 15 (the same d as fp8
//                rows, e8m0 scale 2 c - 1 + j / 4); lane j = 4 of each row
//                loads the seven scale bytes (576 .. 583);
//   bf16 rows    bytes 256 c + 16 j and 256 c + 128 + 16 j: unit j of
//                d-blocks 2 c and 2 c + 1, copied as they are (chunks 2 and
//                3 are loaded into the registers of chunks 0 and 1 once
//                those are stored: a whole bf16 tile would not fit).
template <int kFmt>
__device__ void worker_role(const qsfm_params& p, const Smem& sm, Range rg, int T, uint32_t tmem,
                            const Workspace& ws, int c_idx, int* fault) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // softmax / epilogue view
  const int qd = warp & 3;             // tensor-memory lane quadrant
  const int h0 = kHPT * (warp >> 2);   // first of this warp's kHPT heads
  const int r = 32 * qd + lane;      // tile row of this thread (softmax)
  const uint32_t lane_base = uint32_t(32 * qd) << 16;
  const uint32_t s_addr = tmem + kTmemS + h0 + lane_base;
  const uint32_t prow_addr = sm.base + kSP + uint32_t(r) * 128;
  float* m_used = sm.f(kSMUsed);
  float* alpha = sm.f(kSAlpha);
  float* inv = sm.f(kSInv);
  float* red = sm.f(kSRed);
  int* valid = reinterpret_cast<int*>(sm.ptr + kSValid);
  // producer view
  const int row_lo = tid >> 3;  // 0 .. kRowStride - 1
  const int j = tid & 7;        // == lane & 7
  const int odd = j >> 2;       // j >= 4 stores its odd 16-B unit first (no bank conflicts)
  const int grp = lane & ~7;    // first lane of this row's group of 8
  const int* rows = reinterpret_cast<const int*>(sm.ptr + kSRows);
  const int* kind = reinterpret_cast<const int*>(sm.ptr + kSRowKind);
  constexpr int kRowB = kv_row_bytes(kFmt);
  const uint4 z = make_uint4(0, 0, 0, 0);

  int pr[kRPT], pr_n[kRPT];    // physical rows of the tile to store next / of the one after
  int kd = 0, kd_n = 0;        // their pools (0 ori, 1 cmp)
  uint2 sc[kRPT], sc_n[kRPT];  // their scales: fp8 scale j (x), packed e8m0 bytes (lane 4)
  uint4 R[4][kRPT];            // raw pieces: [chunk][row] (bf16: [2 (chunk & 1) + half][row])
  uint4 RR[kRPT];              // packed rows: the rope piece of chunk 0
  float rsc[kRPT];             // fp8 rows: the row's prescale 2^-k (f16 range)
  int rsh[kRPT];               // fp8 rows: k

  // Rows of tile n from the ring into (prr, kdd); false at the end mark or
  // on abort.
  auto take_rows = [&](uint32_t n, int (&prr)[kRPT], int& kdd) -> bool {
    const uint32_t slot = n % kRing;
    if (!warp_wait_or_abort(sm, kBarRowsFull + slot, (n / kRing) & 1, fault)) return false;
    kdd = kind[slot];
#pragma unroll
    for (int u = 0; u < kRPT; ++u) prr[u] = rows[slot * kTileRows + row_lo + kRowStride * u];
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.bar(kBarRowsEmpty + slot));
    return kdd >= 0;
  };

  // Loads of raw chunk c of row u of the tile with rows (prr, kdd) (bf16:
  // into the registers of chunk c & 1), and with chunk 0 the row's scales.
  auto load_chunk = [&](int c, int u, const int (&prr)[kRPT], int kdd, uint2 (&scl)[kRPT]) {
    const bool v = prr[u] >= 0;
    const uint8_t* row = static_cast<const uint8_t*>(kdd ? p.cmp_kv : p.ori_kv) + size_t(v ? prr[u] : 0) * kRowB;
    if (c == 0) {
      if constexpr (kFmt == QSFM_KV_FP8_FP32_SCALES) {
        const float* spool = kdd ? p.cmp_scale : p.ori_scale;
        scl[u].x = ldg_pred_u32(spool + size_t(v ? prr[u] : 0) * kScales + j, v);
      } else if constexpr (kFmt == QSFM_KV_PACKED640) {
        scl[u] = (v && j == 4) ? ldg_stream_v2(row + 576) : make_uint2(0, 0);
      }
    }
    if constexpr (kFmt == QSFM_KV_FP8_FP32_SCALES) {
      R[c][u] = v ? ldg_stream_v4(row + 128 * c + 16 * j) : z;
    } else if constexpr (kFmt == QSFM_KV_BF16) {
      R[2 * (c & 1)][u] = v ? ldg_stream_v4(row + 256 * c + 16 * j) : z;
      R[2 * (c & 1) + 1][u] = v ? ldg_stream_v4(row + 256 * c + 128 + 16 * j) : z;
    } else {
      if (c == 0) {
        RR[u] = v ? ldg_stream_v4(row + 16 * j) : z;
        R[0][u] = (v && j < 4) ? ldg_stream_v4(row + 128 + 16 * j) : z;
      } else {
        R[c][u] = v ? ldg_stream_v4(row + 64 + 128 * c + 16 * j) : z;
      }
    }
  };

  // Chunk c of the raw tile, converted to bf16 row by row and stored into
  // its two slabs, then published.
  auto store_chunk = [&](int c) {
    const uint32_t tile = sm.base + kSK;
#pragma unroll
    for (int u = 0; u < kRPT; ++u) {
      const int rr = row_lo + kRowStride * u;
      const uint32_t sw = uint32_t(rr & 7);
      if constexpr (kFmt == QSFM_KV_BF16) {
        const uint32_t unit = (uint32_t(j) ^ sw) << 4;
        sts_v4(tile + (2 * c) * kSlabBytes + rr * 128 + unit, R[2 * (c & 1)][u]);
        sts_v4(tile + (2 * c + 1) * kSlabBytes + rr * 128 + unit, R[2 * (c & 1) + 1][u]);
        continue;
      }
      uint4 lo, hi;
      if constexpr (kFmt == QSFM_KV_FP8_FP32_SCALES) {
        // f16 operands: e4m3 -> f16 is exact, then one f16 multiply by the
        // block's scale times the row's prescale 2^-k
        // (the clamp only acts on rows past 2^22, which are flagged)
        const float s = fminf(__shfl_sync(0xffffffffu, __uint_as_float(sc[u].x), grp | (2 * c + odd)) * rsc[u],
                              65504.f / 448.f);
        dequant16_f16(R[c][u], pack_f16(s, s), lo, hi);
      } else {
        const uint32_t w0 = __shfl_sync(0xffffffffu, sc[u].x, grp | 4);  // scale bytes 0..3
        const uint32_t w1 = __shfl_sync(0xffffffffu, sc[u].y, grp | 4);  // scale bytes 4..6
        if (c == 0) {
          sts_v4(tile + rr * 128 + ((uint32_t(j) ^ sw) << 4), RR[u]);  // rope: d-block 0
          if (j < 4) {
            dequant16(R[0][u], e8m0_value(w0 & 0xFFu), lo, hi);
            const uint32_t rowb = tile + kSlabBytes + rr * 128;  // nope d 64..127: d-block 1
            sts_v4(rowb + ((uint32_t(2 * j) ^ sw) << 4), lo);
            sts_v4(rowb + ((uint32_t(2 * j + 1) ^ sw) << 4), hi);
          }
          continue;
        }
        const int sidx = 2 * c - 1 + odd;
        const uint32_t e = (sidx < 4 ? w0 >> (8 * sidx) : w1 >> (8 * (sidx - 4))) & 0xFFu;
        dequant16(R[c][u], e8m0_value(e), lo, hi);
      }
      const uint32_t rowb = tile + (2 * c + odd) * kSlabBytes + rr * 128;
      const uint32_t c0 = 2 * (j & 3);
      sts_v4(rowb + (((c0 + odd) ^ sw) << 4), odd ? hi : lo);
      sts_v4(rowb + (((c0 + 1 - odd) ^ sw) << 4), odd ? lo : hi);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.bar(kBarFull + c));
  };

  // Tile n from the registers into the tile buffer, chunk c once PV(n - 1)
  // has read it. The rows of tile n + 1 are taken first; as each chunk's
  // registers are stored they are reloaded with the same chunk of tile n + 1
  // (bf16 rows: chunks c + 2 of tile n, then chunks 0 and 1 of tile n + 1),
  // so the loads are issued a chunk at a time and have about a tile's time
  // in flight.
  uint32_t n_store = 0;
  bool have_tile = take_rows(0, pr, kd);
  if (have_tile) {
#pragma unroll
    for (int u = 0; u < kRPT; ++u) {
#pragma unroll
      for (int c = 0; c < (kFmt == QSFM_KV_BF16 ? 2 : 4); ++c) load_chunk(c, u, pr, kd, sc);
    }
  }
  auto store_next = [&]() {
    if (!have_tile) return;
    // this tile's scales were loaded with its chunk 0 a tile ago; taking
    // them over only now keeps the copy from waiting on those loads
    if (n_store > 0) {
#pragma unroll
      for (int u = 0; u < kRPT; ++u) sc[u] = sc_n[u];
    }
    const bool more = take_rows(n_store + 1, pr_n, kd_n);
    if constexpr (kFmt == QSFM_KV_FP8_FP32_SCALES) {
      // Per-row prescale: the smallest k with 448 * max scale * 2^-k <=
      // 2^15, so every dequantised value fits in f16 (k = 0 for any row
      // whose values stay within 2^15). The softmax multiplies the row's
      // logits and its P by 2^k; k <= 7 keeps P inside f16. Computed before
      // the wait for the buffer: it needs only the scales.
#pragma unroll
      for (int u = 0; u < kRPT; ++u) {
        float m = fabsf(__uint_as_float(sc[u].x));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        // k = clamp(ceil(log2(m * 448 / 2^15)), 0, kMaxRowShift) from the
        // exponent field (exact for the power-of-two thresholds)
        const float t = m * (448.f / 32768.f);
        const int e = int((__float_as_uint(t) >> 23) & 0xFFu) - 127;  // t in [2^e, 2^(e+1))
        const bool pow2 = (__float_as_uint(t) & 0x7FFFFFu) == 0u;
        int k = t > 1.f ? (pow2 ? e : e + 1) : 0;
        if (k > kMaxRowShift) {
          if (j == 0) atomicOr(fault, QSFM_FAULT_RANGE);
          k = kMaxRowShift;
        }
        rsh[u] = k;
        rsc[u] = __int_as_float((127 - k) << 23);
      }
    }
    // the tile's valid flags (read by the softmax once chunk 0 is published;
    // every worker has read the previous tile's flags before P was written)
    if (j == 0) {
#pragma unroll
      for (int u = 0; u < kRPT; ++u) {
        int flag = pr[u] >= 0 ? 1 : 0;
        if constexpr (kFmt == QSFM_KV_FP8_FP32_SCALES) flag = pr[u] >= 0 ? rsh[u] + 1 : 0;
        valid[row_lo + kRowStride * u] = flag;
      }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {  // unrolled: the raw registers are indexed by c
      if (n_store > 0 && (c & 1) == 0 &&
          !warp_wait_or_abort(sm, kBarFree + (c >> 1), (n_store - 1) & 1, fault)) {
        have_tile = false;
        return;
      }
      store_chunk(c);
#pragma unroll
      for (int u = 0; u < kRPT; ++u) {
        if constexpr (kFmt == QSFM_KV_BF16) {
          if (c < 2) load_chunk(c + 2, u, pr, kd, sc);
          else if (more) load_chunk(c - 2, u, pr_n, kd_n, sc_n);
        } else {
          if (more) load_chunk(c, u, pr_n, kd_n, sc_n);
        }
      }
    }
    ++n_store;
    have_tile = more;
#pragma unroll
    for (int u = 0; u < kRPT; ++u) pr[u] = pr_n[u];
    kd = kd_n;
  };

  // fp8 rows: q of the next live piece, landed in bf16 by TMA, converted to
  // f16 in place with the exact prescale 2^-kq (kq >= 0, the smallest with
  // max |q| 2^-kq < 2^15); returns the piece's logit factor
  // softmax_scale * log2(e) * 2^kq. Every worker thread converts 16 of the
  // 4096 16-byte units (the swizzle is irrelevant to an elementwise pass).
  uint32_t q_conv = 0;  // conversions done (one per live piece)
  auto convert_q = [&]() -> float {
    warp_wait_or_abort(sm, kBarQFull, q_conv & 1, fault);
    ++q_conv;
    const uint32_t qb = sm.base + kSQ;
    uint32_t mx = 0;  // largest bf16 magnitude bit pattern
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
      const uint4 v = lds_v4(qb + 16 * uint32_t(tid + kWorkThreads * i));
      mx = max(mx, max(max(v.x & 0x7FFFu, (v.x >> 16) & 0x7FFFu), max(v.y & 0x7FFFu, (v.y >> 16) & 0x7FFFu)));
      mx = max(mx, max(max(v.z & 0x7FFFu, (v.z >> 16) & 0x7FFFu), max(v.w & 0x7FFFu, (v.w >> 16) & 0x7FFFu)));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    uint32_t* qred = reinterpret_cast<uint32_t*>(red);
    if (lane == 0) qred[warp] = mx;
    named_sync(kBarWork, kWorkThreads);
#pragma unroll
    for (int w = 0; w < kWorkWarps; ++w) mx = max(mx, qred[w]);
    named_sync(kBarWork, kWorkThreads);  // qred (red) is free again
    // bf16 exponent field e: |q| < 2^(e - 126); kq = max(0, e - 141)
    const int kq = max(0, int((mx >> 7) & 0xFFu) - 141);
    const float f = __int_as_float((127 - kq) << 23);
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
      const uint32_t a = qb + 16 * uint32_t(tid + kWorkThreads * i);
      const uint4 v = lds_v4(a);
      uint4 o;
      o.x = pack_f16(__uint_as_float(v.x << 16) * f, __uint_as_float(v.x & 0xFFFF0000u) * f);
      o.y = pack_f16(__uint_as_float(v.y << 16) * f, __uint_as_float(v.y & 0xFFFF0000u) * f);
      o.z = pack_f16(__uint_as_float(v.z << 16) * f, __uint_as_float(v.z & 0xFFFF0000u) * f);
      o.w = pack_f16(__uint_as_float(v.w << 16) * f, __uint_as_float(v.w & 0xFFFF0000u) * f);
      sts_v4(a, o);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.bar(kBarQReady));
    return p.softmax_scale * kLog2e * __int_as_float((127 + kq) << 23);
  };
  float qk_next = p.softmax_scale * kLog2e;  // logit factor of the next piece (fp8: set by convert_q)

  PieceIter pieces(&p, rg, T);
  uint32_t n = 0, pieces_live = 0;
  int t, lo, hi;
  TokenGeom g;
  bool have = pieces.next(t, g, lo, hi);
  int n_tiles = g.n_tiles;
  while (have) {
    const bool whole = (lo == 0 && hi == n_tiles);
    if constexpr (kF16Ops<kFmt>) {
      // q of this piece, unless it was converted at the end of the last one
      if (lo < hi && q_conv == pieces_live) qk_next = convert_q();
    }
    const float qk_scale = qk_next;
    // this thread's head sink (log2 units); the unit's heads start at unit_head0
    const float sink2 =
        (tid < 64 && p.sinks != nullptr) ? __ldg(p.sinks + unit_head0(p, t) + tid) * kLog2e : -INFINITY;
    const int slot = (t == rg.t0) ? 2 * c_idx : 2 * c_idx + 1;
    const bool writable = whole || slot < ws.slots;  // split pieces need the workspace
    if (!writable && tid == 0) atomicOr(fault, QSFM_FAULT_METADATA);
    // Lane i of the warp keeps the running sum of P for head h0 + i % kHPT
    // over this warp's 32 rows: each tile's P is folded in with a lane
    // reduction once P is published (one register instead of kHPT).
    float l_sum = 0.f;
    if (tid < 64) m_used[tid] = -INFINITY;
    named_sync(kBarWork, kWorkThreads);
    // One call site for the tile stores (the code stays small): the next
    // tile goes into the buffer at the top of each iteration, as PV(n - 1)
    // frees it; tile 0 right after the first q conversion (q lands first).
    bool pending = n_store == 0;
#pragma unroll 1
    for (int k = lo;; ++k) {
      if (pending) store_next();
      if (k >= hi) break;
      pending = true;
      const uint32_t par = n & 1;
      // Lane 0 of each warp polls. After an abort the waits fall through at
      // once; the workers keep running the same named-barrier sequence so
      // that none of them blocks.
      warp_wait_or_abort(sm, kBarFull + 0, par, fault);  // the tile's valid flags
      const int vflag = valid[r];
      const bool v = vflag != 0;
      // fp8 rows: the row's values were prescaled by 2^-k (flag = k + 1)
      const float fr = kF16Ops<kFmt> && v ? __int_as_float((126 + vflag) << 23) : 1.f;
      const float qk_row = qk_scale * fr;
      warp_wait_or_abort(sm, kBarSFull, par, fault);
      tc_fence_after();
      float x[kHPT];
      tmem_load(s_addr, x);
      tmem_ld_wait();
      bool move = true;  // the first tile of a piece always sets the max
      if (k != lo) {
        // Fast path: t = score * scale - m (log2 units), P = 2^t computed
        // before the vote; valid only if no t exceeds 8 anywhere in the tile.
        float tmax = -INFINITY;
#pragma unroll
        for (int i = 0; i < kHPT; i += 4) {
          const float4 m4 = *reinterpret_cast<const float4*>(m_used + h0 + i);
          const float t0 = v ? fmaf(x[i], qk_row, -m4.x) : -INFINITY;
          const float t1 = v ? fmaf(x[i + 1], qk_row, -m4.y) : -INFINITY;
          const float t2 = v ? fmaf(x[i + 2], qk_row, -m4.z) : -INFINITY;
          const float t3 = v ? fmaf(x[i + 3], qk_row, -m4.w) : -INFINITY;
          tmax = fmaxf(tmax, fmaxf(fmaxf(t0, t1), fmaxf(t2, t3)));
          x[i] = ex2_approx(t0);
          x[i + 1] = ex2_approx(t1);
          x[i + 2] = ex2_approx(t2);
          x[i + 3] = ex2_approx(t3);
        }
        move = named_sync_or(kBarWork, kWorkThreads, tmax > kRescaleLog2);  // also true against -inf
      }
      float lscale = 1.f;  // 0 after a moved max: the running sums take alpha first
      if (move) {
        // Slow path: the scores again, the tile max per head over its 128
        // rows, the new running max, then O^T and the row sums rescaled.
        if (k != lo) {
          tmem_load(s_addr, x);
          tmem_ld_wait();
        }
#pragma unroll
        for (int i = 0; i < kHPT; ++i) x[i] = v ? x[i] * qk_row : -INFINITY;
        const float mx = reduce_lanes<true>(x);  // head h0 + lane % kHPT, this quadrant's rows
        if (lane < kHPT) red[qd * 64 + h0 + lane] = mx;
        named_sync(kBarWork, kWorkThreads);
        if (tid < 64) {
          const float mt = fmaxf(fmaxf(red[tid], red[64 + tid]), fmaxf(red[128 + tid], red[192 + tid]));
          const float mu = m_used[tid];
          float a = 1.f;
          if (mt > -INFINITY && (mu == -INFINITY || mt > mu + kRescaleLog2)) {
            a = (mu == -INFINITY) ? 0.f : exp2f(mu - mt);
            m_used[tid] = mt;
          }
          alpha[tid] = a;
        }
        named_sync(kBarWork, kWorkThreads);
        if (k != lo) {
          // O^T at this thread's lane, its kHPT heads, every chunk. The PV
          // products of the earlier tiles have completed: S^T(n) was
          // committed after them.
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float o[kHPT];
            const uint32_t addr = tmem + kTmemO + 64 * c + h0 + lane_base;
            tmem_load(addr, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < kHPT; ++i) o[i] *= alpha[h0 + i];
            tmem_store(addr, o);
          }
          tmem_st_wait();
        }
        tmem_load(s_addr, x);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < kHPT; ++i) {
          const float m = m_used[h0 + i];
          const float mz = m == -INFINITY ? 0.f : m;
          x[i] = ex2_approx(v ? fmaf(x[i], qk_row, -mz) : -INFINITY);
        }
        lscale = 0.f;
      }
      // P into the P buffer as [128 rows][64 heads] bf16 with the 128-B
      // swizzle (the MN-major B operand of PV): this thread's row, its
      // 16-byte units of 8 heads
#pragma unroll
      for (int vv = 0; vv < kHPT / 8; ++vv) {
        const uint32_t u = uint32_t((h0 >> 3) + vv);
        uint4 pk;
        if constexpr (kF16Ops<kFmt>) {
          // P times the row factor (the row's V~ values carry 2^-k)
          pk.x = pack_f16(x[8 * vv + 0] * fr, x[8 * vv + 1] * fr);
          pk.y = pack_f16(x[8 * vv + 2] * fr, x[8 * vv + 3] * fr);
          pk.z = pack_f16(x[8 * vv + 4] * fr, x[8 * vv + 5] * fr);
          pk.w = pack_f16(x[8 * vv + 6] * fr, x[8 * vv + 7] * fr);
        } else {
          pk.x = pack_bf16(x[8 * vv + 0], x[8 * vv + 1]);
          pk.y = pack_bf16(x[8 * vv + 2], x[8 * vv + 3]);
          pk.z = pack_bf16(x[8 * vv + 4], x[8 * vv + 5]);
          pk.w = pack_bf16(x[8 * vv + 6], x[8 * vv + 7]);
        }
        sts_v4(prow_addr + ((u ^ uint32_t(r & 7)) << 4), pk);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.bar(kBarPFull));
      {
        // running sums += this tile's P, folded over the warp's rows (after
        // P is published: off the PV path); a moved max rescales them first
        const float tile_sum = reduce_lanes<false>(x);
        if (lscale == 0.f) l_sum *= alpha[h0 + (lane % kHPT)];
        l_sum += tile_sum;
      }
      ++n;
    }
    // The next piece's geometry, read now: its loads overlap the wait for
    // this piece's last PV product.
    int t_next = 0, lo_next = 0, hi_next = 0;
    const bool have_next = pieces.next(t_next, g, lo_next, hi_next);
    const int n_tiles_next = g.n_tiles;
    if constexpr (kF16Ops<kFmt>) {
      // the next piece's q before this epilogue, so that its first QK^T
      // does not wait for the epilogue
      if (have_next && lo_next < hi_next && lo < hi) qk_next = convert_q();
    }
    // ---------------- epilogue of the piece
    const bool any = lo < hi;
    if (any && lane < kHPT) red[qd * 64 + h0 + lane] = l_sum;
    named_sync(kBarWork, kWorkThreads);
    if (tid < 64 && writable) {
      const float lt = any ? (red[tid] + red[64 + tid]) + (red[128 + tid] + red[192 + tid]) : 0.f;
      const float mu = m_used[tid];
      const float lse2 = lt > 0.f ? mu + log2f(lt) : -INFINITY;
      if (whole) {
        float den = lt;
        if (p.sinks != nullptr && lt > 0.f) den += exp2f(sink2 - mu);
        inv[tid] = lt > 0.f ? 1.f / den : 0.f;
        if (p.return_lse) p.softmax_lse[size_t(t) * 64 + tid] = lse2 * kLn2;
      } else {
        inv[tid] = lt > 0.f ? 1.f / lt : 0.f;
        ws.lse[size_t(slot) * 64 + tid] = lse2 * kLn2;
      }
    }
    named_sync(kBarWork, kWorkThreads);
    // O^T chunk by chunk once the last PV product has completed it: this
    // thread holds head-dim element d = 128 c + 32 qd + lane of its kHPT
    // heads. Whole units: the two lanes of a pair swap values so that each
    // stores two adjacent d (4 bytes) of kHPT / 2 heads; a warp writes 64
    // contiguous bytes per head. Split pieces store fp32 rows (128 bytes per
    // head per warp).
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      float o[kHPT];
      if (any) {
        if ((c & 1) == 0) warp_wait_or_abort(sm, kBarFree + (c >> 1), (n - 1) & 1, fault);
        tc_fence_after();
        tmem_load(tmem + kTmemO + 64 * c + h0 + lane_base, o);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < kHPT; i += 4) {
          const float4 iv = *reinterpret_cast<const float4*>(inv + h0 + i);
          o[i] *= iv.x;
          o[i + 1] *= iv.y;
          o[i + 2] *= iv.z;
          o[i + 3] *= iv.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < kHPT; ++i) o[i] = 0.f;
      }
      const int d = 128 * c + 32 * qd + lane;
      if (whole) {
        const int od = lane & 1;
        uint32_t* out = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(p.attn_out) +
                                                    (size_t(t) * 64 + h0 + od) * kDim + (d & ~1));
#pragma unroll
        for (int i = 0; i < kHPT / 2; ++i) {
          const float send = od ? o[2 * i] : o[2 * i + 1];
          const float got = __shfl_xor_sync(0xffffffffu, send, 1);
          const float lo_v = od ? got : o[2 * i];
          const float hi_v = od ? o[2 * i + 1] : got;
          out[size_t(2 * i) * (kDim / 2)] = pack_bf16(lo_v, hi_v);
        }
      } else if (writable) {
        float* out = ws.out + (size_t(slot) * 64 + h0) * kDim + d;
#pragma unroll
        for (int i = 0; i < kHPT; ++i) out[size_t(i) * kDim] = o[i];
      }
    }
    if (any) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.bar(kBarOFree));
      ++pieces_live;
    }
    named_sync(kBarWork, kWorkThreads);  // m_used / inv / red are reused by the next piece
    if (*sm.abort_flag()) break;         // uniform: read after the barrier
    have = have_next;
    t = t_next;
    lo = lo_next;
    hi = hi_next;
    n_tiles = n_tiles_next;
  }
}

// Runs before the plan is readable, while the plan kernel still runs: warms
// L2 with the Q and the sparse-index row of the unit this CTA most likely
// starts with (the plan cuts equal-cost units evenly, so CTA c of G starts
// near unit c T / G). Prefetches only, no loads to wait for, no fault bits:
// a wrong guess costs bandwidth, never results or time.
__device__ __forceinline__ void warm_first_token(const qsfm_params& p, int T, int c, int G, int lane) {
  const int t = int((long long)c * T / G);
  if (t >= T) return;
  if (lane == 0)
    bulk_prefetch_l2(static_cast<const uint8_t*>(p.q) + size_t(t) * kHeads * kDim * 2, kHeads * kDim * 2);
  if (p.cmp_sparse_indices != nullptr) {
    const uint8_t* ix = reinterpret_cast<const uint8_t*>(p.cmp_sparse_indices + size_t(t >> unit_shift(p)) * p.k2);
    for (int off = 128 * lane; off < 4 * p.k2; off += 32 * 128) prefetch_l2(ix + off);
  }
}

template <int kFmt>
__global__ void __launch_bounds__(kThreads, 1)
    attention_kernel(const qsfm_params p, const int T, const Workspace ws, int* fault,
                     const __grid_constant__ CUtensorMap qmap) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  Smem sm;
  sm.base = (raw_addr + 1023u) & ~1023u;
  sm.ptr = smem_raw + (sm.base - raw_addr);

  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) warm_first_token(p, T, blockIdx.x, gridDim.x, tid);
  grid_dependency_wait();    // the plan (and every input) is written by now
  grid_launch_dependents();  // the combine kernel may take SMs as CTAs finish
  const int* meta = p.metadata;
  if (meta[0] != kMetaMagic || meta[2] != T) {
    if (tid == 0 && blockIdx.x == 0) atomicOr(fault, QSFM_FAULT_METADATA);
    return;
  }
  const int G = meta[1];
  if (G < 0 || G > int(gridDim.x) || G > QSFM_MAX_CTAS) {
    if (tid == 0 && blockIdx.x == 0) atomicOr(fault, QSFM_FAULT_METADATA);
    return;
  }
  const int c = blockIdx.x;
  if (c >= G) return;
  const Range rg{meta[kMetaHeader + 2 * c], meta[kMetaHeader + 2 * c + 1],
                 meta[kMetaHeader + 2 * c + 2], meta[kMetaHeader + 2 * c + 3]};
  if (rg.t0 < 0 || rg.t1 > T || rg.t0 > rg.t1 || rg.k0 < 0 || rg.k1 < 0 ||
      (rg.t1 == T && rg.k1 != 0)) {
    if (tid == 0) atomicOr(fault, QSFM_FAULT_METADATA);
    return;
  }
  if (rg.t0 == rg.t1 && rg.k0 == rg.k1) return;

  if (tid == 0) {
    mbar_init(sm.bar(kBarQFull), 1);
    for (int i = 0; i < 4; ++i) mbar_init(sm.bar(kBarFull + i), kWorkWarps);
    for (int i = 0; i < 2; ++i) mbar_init(sm.bar(kBarFree + i), 1);
    mbar_init(sm.bar(kBarSFull), 1);
    mbar_init(sm.bar(kBarPFull), kWorkWarps);
    mbar_init(sm.bar(kBarOFree), kWorkWarps);
    for (int i = 0; i < kRing; ++i) {
      mbar_init(sm.bar(kBarRowsFull + i), 1);
      mbar_init(sm.bar(kBarRowsEmpty + i), kWorkWarps);
    }
    mbar_init(sm.bar(kBarDrain), 1);
    mbar_init(sm.bar(kBarQReady), kWorkWarps);
    *sm.abort_flag() = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(sm.tmem_slot(), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_slot();

  if (warp < kWorkWarps) {
    worker_role<kFmt>(p, sm, rg, T, tmem, ws, c, fault);
  } else if (warp == kMmaWarp) {
    mma_role<kFmt>(p, sm, rg, T, tmem, &qmap, fault);
    if ((tid & 31) == 0) {
      // every MMA issued above has completed before tensor memory is freed
      // (after an abort some may still be in flight)
      mma_commit(sm.bar(kBarDrain));
      wait_or_abort(sm, kBarDrain, 0, fault);
    }
  } else {
    resolver_role<kFmt>(p, sm, rg, T, fault);
  }

  // Roles run on single lanes (the MMA issue): each warp's lanes meet before
  // the barrier (a barrier reached by part of a warp counts the whole warp).
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Tensor map of q viewed as [T * 64 rows, 512 bf16 columns], boxes of
// 64 rows x 64 columns (128 B) with the 128-B swizzle of the MMA operand.
cudaError_t make_q_map(const void* q, int T, CUtensorMap* map) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult qres;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &qres) == cudaSuccess &&
        qres == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (encode == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cuuint64_t(kDim), cuuint64_t(T) * kHeads};
  const cuuint64_t strides[1] = {cuuint64_t(kDim) * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), dims,
                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_attention(const qsfm_params& p, int num_tokens, int num_ctas,
                             const Workspace& ws, int* fault, cudaStream_t s) {
  // one instantiation per KV row format, so none pays for the others
  auto* kernel = p.kv_layout == QSFM_KV_PACKED640 ? attention_kernel<QSFM_KV_PACKED640>
                 : p.kv_layout == QSFM_KV_BF16    ? attention_kernel<QSFM_KV_BF16>
                                                  : attention_kernel<QSFM_KV_FP8_FP32_SCALES>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
  if (e != cudaSuccess) return e;
  CUtensorMap qmap;
  e = make_q_map(p.q, num_tokens, &qmap);
  if (e != cudaSuccess) return e;
  return launch_after_predecessor(kernel, dim3(num_ctas), dim3(kThreads), kSmemAlloc, s, p, num_tokens,
                                  ws, fault, qmap);
}

}  // namespace qsfm
