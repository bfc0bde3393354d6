// Attention kernel of the quantized shared-KV sparse MLA forward (sm_103a).
//
// Computes, for every planned (token, KV-tile range) piece,
//   O = softmax([Q K~^T * softmax_scale, sink]) V~  with K~ = V~
// (QuantSparseFlashMla, function description formula; sink from its
// parameter table row "sinks"; lse from KvQuantSparseAttnSharedKv, parameter
// table row softmax_lse).
//
// Orientation. The contractions run transposed so that the KV rows of a tile
// (64 rows) are the M dimension of the score product and the 64 heads are N:
//   S^T[j, h]  = sum_d K~[j, d] Q[h, d]      (M = 64 rows, N = 64, K = 512)
//   O^T[d, h] += sum_j V~[j, d] P[h, j]      (M = 128 d per chunk, N = 64,
//                                             K = 64 rows, 4 chunks)
// Both accumulators live in tensor memory: S^T in two buffers of 64 columns
// (an M = 64 accumulator fills lanes 0-15 of each 32-lane quarter), O^T in
// 256 columns. One dequantised bf16 tile (64 rows x 512, 128-B swizzle, 8
// d-blocks of 8 KB) is the K-major A operand of the first product and, read
// through an MN-major descriptor, the A operand of the second.
//
// Pipeline. Two tile stages in shared memory: while the tensor cores and the
// softmax work on tile n, the producers fill the other stage with tile n+1.
// Two threads issue the tensor-core work, each in its own order: QK^T of a
// tile chunk by chunk as the producers publish it, PV of a tile once the
// softmax has written P. So QK^T(n+1) runs while the softmax works on tile
// n, and PV(n) while the producers fill tile n+2's stage. Before the plan is
// readable (the plan kernel may still run), the producer warps warm L2 with
// the inputs of the token the CTA most likely starts with.
//
// Warp roles (15 warps; at most 4 per SM sub-partition, so 128 registers):
//   warps 0-3   softmax + epilogue. Warp q owns tile rows 16q..16q+15; each
//               thread holds two rows x 16 heads of S^T (the accumulator-
//               fragment layout), keeps the row sums of its 16 heads in
//               registers and writes its P values with stmatrix. In the
//               epilogue thread i owns head-dim lane i of O^T.
//   warps 4-11  producers: take a tile's physical rows from the resolver,
//               load their fp8 bytes and scales into registers, dequantise
//               the whole tile into registers, start the next tile's loads,
//               then store the tile chunk by chunk (a chunk = 64 rows x 128 d
//               = 2 d-blocks) once its stage is free. Packed 640-byte rows
//               and bf16 rows have producers of their own (one kernel
//               instantiation per row format); the tile they store is the
//               same.
//   warp 12     QK^T issue (one thread): Q by TMA, QK^T chunk by chunk as the
//               producers publish the chunks.
//   warp 14     PV issue (one thread): PV once the softmax has written P, and
//               the commits that release stages and hand O^T to the epilogue.
//   warp 13     resolver: runs up to 4 tiles ahead, turns each tile's slots
//               into physical rows (sparse indices, block tables) in a
//               shared-memory ring, and asks L2 for those rows' bytes.
// mbarriers carry every hand-off; every wait is bounded in time.
//
// Softmax: the running max m_used per head is moved only when a tile's max
// exceeds it by more than 8 (log2 units); a named-barrier vote detects that
// case, so most tiles need no cross-thread max reduction. When it moves, O^T
// and the row sums l are rescaled exactly. P <= 2^8 in bf16.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "qsfm_device.cuh"
#include "qsfm_internal.h"

namespace qsfm {
namespace {

static_assert(kTileRows == 64, "the kernel's layouts assume 64-row tiles");

constexpr int kSoftWarps = 4;
constexpr int kProdWarps = 8;
constexpr int kMmaWarp = kSoftWarps + kProdWarps;
constexpr int kResolverWarp = kMmaWarp + 1;
constexpr int kPvWarp = kResolverWarp + 1;
constexpr int kThreads = (kPvWarp + 1) * 32;
constexpr int kRing = 4;  // tiles of resolved rows in flight
constexpr int kSoftThreads = kSoftWarps * 32;
constexpr int kBarSoft = 1;  // named barrier id of the softmax warps
constexpr int kStages = 2;

// shared memory map (byte offsets from a 1024-aligned base)
constexpr uint32_t kDBlockBytes = kTileRows * 128;           // 64 rows x 64 d (bf16)
constexpr uint32_t kStageBytes = 8 * kDBlockBytes;           // one tile: 64 KB
constexpr uint32_t kPBytes = kTileRows * 128;                // P: 64 rows x 64 heads (bf16)
constexpr uint32_t kSK = 0;                                  // K~ stages
constexpr uint32_t kSQ = kSK + kStages * kStageBytes;        // Q: 8 d-blocks x 64 heads x 128 B
constexpr uint32_t kSP = kSQ + 8 * 64 * 128;                 // P stages
constexpr uint32_t kSRed = kSP + kStages * kPBytes;          // [4][64] f32 per-warp partials
constexpr uint32_t kSMUsed = kSRed + 1024;                   // [64] f32
constexpr uint32_t kSAlpha = kSMUsed + 256;                  // [64] f32
constexpr uint32_t kSInv = kSAlpha + 256;                    // [64] f32
constexpr uint32_t kSValid = kSInv + 256;                    // [2][64] i32
constexpr uint32_t kSRows = kSValid + 512;                   // [kRing][64] i32 physical rows
constexpr uint32_t kSRowKind = kSRows + kRing * kTileRows * 4;  // [kRing] i32: 0 ori, 1 cmp, -1 end
constexpr uint32_t kSBar = kSRowKind + 64;                   // mbarriers, tmem base, flags
constexpr uint32_t kSmemBytes = kSBar + 256;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;

// mbarrier slots
constexpr int kBarQFull = 0;
constexpr int kBarKvFull = 1;    // [stage][chunk], one arrive per producer warp
constexpr int kBarKvEmpty = 9;   // [stage]: the PV product of the stage's tile completed
constexpr int kBarSFull = 11;    // [stage]
constexpr int kBarSFree = 13;    // [stage]
constexpr int kBarPFull = 15;    // [stage]
constexpr int kBarODone = 17;
constexpr int kBarOFree = 18;
constexpr int kBarRowsFull = 19;   // [ring slot]
constexpr int kBarRowsEmpty = 23;  // [ring slot], one arrive per producer warp
constexpr int kNumBars = 27;
static_assert(kNumBars * 8 <= 224, "barriers overlap the tmem slot");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;  // + 64 * stage
constexpr uint32_t kTmemO = 256;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kIdescQK = make_idesc_bf16(64, 64, /*a_mn=*/0, /*b_mn=*/0);
constexpr uint32_t kIdescPV = make_idesc_bf16(128, 64, /*a_mn=*/1, /*b_mn=*/1);
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait

struct Range {
  int t0, k0, t1, k1;
};

// Walks the (token, tile-range) pieces of a CTA's range in order.
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

// Walks the (token, tile) jobs of the range, skipping tokens without tiles.
struct JobIter {
  PieceIter pieces;
  int tok = -1, k = 0, hi = 0;
  TokenGeom g;
  __device__ JobIter(const qsfm_params* p, Range r, int T) : pieces(p, r, T) {}
  __device__ bool next(int& tok_out, int& k_out, TokenGeom& g_out) {
    while (tok < 0 || k >= hi) {
      int lo;
      if (!pieces.next(tok, g, lo, hi)) return false;
      k = lo;
    }
    tok_out = tok;
    k_out = k++;
    g_out = g;
    return true;
  }
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Max (kMax) or sum of 16 values per lane over the 8 lanes of a warp that
// share lane % 4 (lane bits 2-4). Afterwards lane l holds, in v[0] and v[1],
// the results for value indices 2 * (l >> 2) and 2 * (l >> 2) + 1.
template <bool kMax>
__device__ __forceinline__ void reduce_rows16(float (&v)[16]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int w = 16, n = 8; w >= 4; w >>= 1, n >>= 1) {
    const bool up = lane & w;
#pragma unroll
    for (int i = 0; i < n; ++i) {
      const float keep = up ? v[n + i] : v[i];
      const float send = up ? v[i] : v[n + i];
      const float got = __shfl_xor_sync(0xffffffffu, send, w);
      v[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
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

// ------------------------------------------------------------- resolver
// Tile n's rows go to ring slot n % kRing: 64 physical rows (block * 128 +
// offset, -1 = masked) and the pool they come from. After the CTA's last tile
// the resolver writes an end mark (-1) in the next slot.
template <int kFmt>
__device__ void resolver_role(const qsfm_params& p, const Smem& sm, Range rg, int T, int* fault) {
  const int lane = threadIdx.x & 31;
  int* rows = reinterpret_cast<int*>(sm.ptr + kSRows);
  int* kind = reinterpret_cast<int*>(sm.ptr + kSRowKind);
  JobIter jobs(&p, rg, T);
  int tok, k, last_tok = -1;
  TokenGeom g;
  for (uint32_t n = 0;; ++n) {
    const bool more = jobs.next(tok, k, g);
    const uint32_t slot = n % kRing;
    if (!warp_wait_or_abort(sm, kBarRowsEmpty + slot, ((n / kRing) & 1) ^ 1, fault)) return;
    if (!more) {
      if (lane == 0) kind[slot] = -1;
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.bar(kBarRowsFull + slot));
      return;
    }
    if (g.tok != last_tok) {
      // the next token's index list goes to L2 while this token is resolved
      if (p.cmp_sparse_indices != nullptr && g.tok + 1 < (T >> unit_shift(p))) {
        const uint8_t* ix = reinterpret_cast<const uint8_t*>(p.cmp_sparse_indices + (size_t)(g.tok + 1) * p.k2);
        for (int off = 128 * lane; off < 4 * p.k2; off += 32 * 128) prefetch_l2(ix + off);
      }
      last_tok = g.tok;
    }
    const int cmp = k >= g.ori_tiles ? 1 : 0;
    int pr[2];
    resolve_two(p, g, k, lane, fault, pr);
    const uint8_t* pool = static_cast<const uint8_t*>(cmp ? p.cmp_kv : p.ori_kv);
    const float* spool = cmp ? p.cmp_scale : p.ori_scale;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      rows[slot * kTileRows + lane + 32 * u] = pr[u];
      if (pr[u] >= 0) {
        if constexpr (kFmt == QSFM_KV_PACKED640) {
          const uint8_t* src = pool + size_t(pr[u]) * QSFM_PACKED_ROW_BYTES;
#pragma unroll
          for (int c = 0; c < 5; ++c) prefetch_l2(src + 128 * c);
        } else if constexpr (kFmt == QSFM_KV_BF16) {
          const uint8_t* src = pool + size_t(pr[u]) * QSFM_BF16_ROW_BYTES;
#pragma unroll
          for (int c = 0; c < 8; ++c) prefetch_l2(src + 128 * c);
        } else {
          const uint8_t* src = pool + size_t(pr[u]) * kDim;
#pragma unroll
          for (int c = 0; c < 4; ++c) prefetch_l2(src + 128 * c);
          prefetch_l2(spool + size_t(pr[u]) * kScales);
        }
      }
    }
    if (lane == 0) kind[slot] = cmp;
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.bar(kBarRowsFull + slot));
  }
}

// ------------------------------------------------------------- producers
// Thread (row_lo, j) of the 8 producer warps: tile rows row_lo and row_lo +
// 32, 16-byte slot j of each 128-byte chunk of those rows.
__device__ void producer_role(const qsfm_params& p, const Smem& sm, int* fault) {
  const int ptid = threadIdx.x - kSoftThreads;  // 0..255 (8 producer warps)
  const int lane = threadIdx.x & 31;
  const int row_lo = ptid >> 3;   // 0..31
  const int j = ptid & 7;
  const int odd_first = j >> 2;   // j >= 4 stores its odd 16-B chunk first (no bank conflicts)
  const int* rows = reinterpret_cast<const int*>(sm.ptr + kSRows);
  const int* kind = reinterpret_cast<const int*>(sm.ptr + kSRowKind);

  int pr[2];
  float csc[2];  // scale j of each row (this lane's share of the row's 8 scales)
  uint4 R0[2], R1[2], R2[2], R3[2];  // fp8 bytes of chunks 0..3 of the two rows

  // Rows of tile n from the ring; their loads start at once. False at the
  // end mark or on abort.
  auto fetch = [&](uint32_t n) -> bool {
    const uint32_t slot = n % kRing;
    if (!warp_wait_or_abort(sm, kBarRowsFull + slot, (n / kRing) & 1, fault)) return false;
    const int kd = kind[slot];
    pr[0] = rows[slot * kTileRows + row_lo];
    pr[1] = rows[slot * kTileRows + row_lo + 32];
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.bar(kBarRowsEmpty + slot));
    if (kd < 0) return false;
    const uint8_t* pool = static_cast<const uint8_t*>(kd ? p.cmp_kv : p.ori_kv);
    const float* spool = kd ? p.cmp_scale : p.ori_scale;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const bool v = pr[u] >= 0;
      const uint8_t* src = pool + size_t(v ? pr[u] : 0) * kDim + 16 * j;
      R0[u] = v ? ldg_stream_v4(src) : make_uint4(0, 0, 0, 0);
      R1[u] = v ? ldg_stream_v4(src + 128) : make_uint4(0, 0, 0, 0);
      R2[u] = v ? ldg_stream_v4(src + 256) : make_uint4(0, 0, 0, 0);
      R3[u] = v ? ldg_stream_v4(src + 384) : make_uint4(0, 0, 0, 0);
      csc[u] = v ? __ldg(spool + size_t(pr[u]) * kScales + j) : 0.f;
    }
    return true;
  };

  // Per tile: dequantise it into registers (this waits for its loads), start
  // the next tile's loads, then wait for the stage and store. The next
  // tile's loads are in flight during the stage wait and the stores.
  bool have = fetch(0);
  for (uint32_t n = 0; have; ++n) {
    const uint32_t st = n & 1;
    uint4 D[4][2][2];  // [chunk][row][16-byte half], bf16
    const int vrow0 = pr[0] >= 0, vrow1 = pr[1] >= 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int src_lane = (lane & ~7) | (2 * c + (j >> 2));
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float sc = __shfl_sync(0xffffffffu, csc[u], src_lane);
        const uint4 raw = c == 0 ? R0[u] : c == 1 ? R1[u] : c == 2 ? R2[u] : R3[u];
        // packed fp32 multiplies: 3 % faster here (the packed-row producer
        // keeps dequant16: there they were 2.5 % slower)
        dequant16_x2(raw, sc, D[c][u][0], D[c][u][1]);
      }
    }
    have = fetch(n + 1);
    if (!warp_wait_or_abort(sm, kBarKvEmpty + st, ((n >> 1) & 1) ^ 1, fault)) return;
    const uint32_t stage = sm.base + kSK + st * kStageBytes;
    if (j == 0) {
      int* valid = reinterpret_cast<int*>(sm.ptr + kSValid) + st * kTileRows;
      valid[row_lo] = vrow0;
      valid[row_lo + 32] = vrow1;
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t blk = stage + (2 * c + (j >> 2)) * kDBlockBytes;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int r = row_lo + 32 * u;
        const uint32_t sw = uint32_t(r & 7);
        const uint32_t rowb = blk + r * 128;
        const uint32_t c0 = 2 * (j & 3);
        sts_v4(rowb + (((c0 + odd_first) ^ sw) << 4), odd_first ? D[c][u][1] : D[c][u][0]);
        sts_v4(rowb + (((c0 + 1 - odd_first) ^ sw) << 4), odd_first ? D[c][u][0] : D[c][u][1]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.bar(kBarKvFull + 4 * st + c));
    }
  }
}

// Producers for packed 640-byte rows (bf16 rope, bytes 0..127 | e4m3fn nope,
// bytes 128..575 | e8m0 scales, bytes 576..582 | pad; KvQuantSparseAttnSharedKv
// constraints). The tile in shared memory is the same as for fp8 rows: d 0..63
// (d-block 0) is the rope, d 64..511 the nope. Thread (row_lo, j): rows
// row_lo and row_lo + 32; of each row the 16-byte pieces j (rope elements
// 8j .. 8j + 7, copied as they are) and 8 + m for m = 8i + j, i = 0..3
// (nope elements 16m .. 16m + 15 of d-block 1 + m / 4 with scale m / 4;
// i = 3 only for j < 4). Lane j = 4 of each row also loads the piece with
// the seven scale bytes. Nope piece m lands in chunk (1 + 2i + j / 4) / 2:
// chunk i for j < 4, chunk i + 1 for j >= 4. The loads of a tile are issued
// after the previous tile is stored (the registers hold one tile).
__device__ __forceinline__ float e8m0_value(uint32_t e) {
  // 2^(e - 127): the fp32 with biased exponent e (e = 0: the subnormal 2^-127)
  return e == 0xFFu ? __uint_as_float(0x7FC00000u) : e == 0u ? __uint_as_float(0x00400000u)
                                                             : __uint_as_float(e << 23);
}

__device__ void producer_role_packed(const qsfm_params& p, const Smem& sm, int* fault) {
  const int ptid = threadIdx.x - kSoftThreads;  // 0..255 (8 producer warps)
  const int lane = threadIdx.x & 31;
  const int row_lo = ptid >> 3;  // 0..31
  const int j = ptid & 7;
  const int odd_first = j >> 2;  // j >= 4 stores its odd 16-B unit first (no bank conflicts)
  const int* rows = reinterpret_cast<const int*>(sm.ptr + kSRows);
  const int* kind = reinterpret_cast<const int*>(sm.ptr + kSRowKind);
  constexpr int kRow = QSFM_PACKED_ROW_BYTES;

  int pr[2];
  uint4 Rr[2];     // rope piece j of each row (bf16)
  uint4 Rn[4][2];  // nope pieces m = 8i + j (e4m3fn)
  uint4 Rs[2];     // scale piece (lane j = 4 only)

  auto fetch = [&](uint32_t n) -> bool {
    const uint32_t slot = n % kRing;
    if (!warp_wait_or_abort(sm, kBarRowsFull + slot, (n / kRing) & 1, fault)) return false;
    const int kd = kind[slot];
    pr[0] = rows[slot * kTileRows + row_lo];
    pr[1] = rows[slot * kTileRows + row_lo + 32];
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.bar(kBarRowsEmpty + slot));
    if (kd < 0) return false;
    const uint8_t* pool = static_cast<const uint8_t*>(kd ? p.cmp_kv : p.ori_kv);
    const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const bool v = pr[u] >= 0;
      const uint8_t* base = pool + size_t(v ? pr[u] : 0) * kRow;
      Rr[u] = v ? ldg_stream_v4(base + 16 * j) : z;
#pragma unroll
      for (int i = 0; i < 3; ++i) Rn[i][u] = v ? ldg_stream_v4(base + 128 + 16 * (8 * i + j)) : z;
      Rn[3][u] = (v && j < 4) ? ldg_stream_v4(base + 128 + 16 * (24 + j)) : z;
      Rs[u] = (v && j == 4) ? ldg_stream_v4(base + 576) : z;
    }
    return true;
  };

  for (uint32_t n = 0; fetch(n); ++n) {
    const uint32_t st = n & 1;
    uint4 D[4][2][2];  // [i][row][16-byte half] of nope piece 8i + j, bf16
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint32_t w0 = __shfl_sync(0xffffffffu, Rs[u].x, (lane & ~7) | 4);  // scale bytes 0..3
      const uint32_t w1 = __shfl_sync(0xffffffffu, Rs[u].y, (lane & ~7) | 4);  // scale bytes 4..6
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int sidx = 2 * i + (j >> 2);  // scale of nope piece 8i + j
        const uint32_t e = (sidx < 4 ? w0 >> (8 * sidx) : w1 >> (8 * (sidx - 4))) & 0xFFu;
        dequant16(Rn[i][u], e8m0_value(e), D[i][u][0], D[i][u][1]);
      }
    }
    if (!warp_wait_or_abort(sm, kBarKvEmpty + st, ((n >> 1) & 1) ^ 1, fault)) return;
    const uint32_t stage = sm.base + kSK + st * kStageBytes;
    if (j == 0) {
      int* valid = reinterpret_cast<int*>(sm.ptr + kSValid) + st * kTileRows;
      valid[row_lo] = pr[0] >= 0;
      valid[row_lo + 32] = pr[1] >= 0;
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int r = row_lo + 32 * u;
        const uint32_t sw = uint32_t(r & 7);
        if (c == 0) sts_v4(stage + r * 128 + ((uint32_t(j) ^ sw) << 4), Rr[u]);  // rope: d-block 0
        // nope piece of this chunk: i = c (j < 4) or i = c - 1 (j >= 4)
        const bool has = j < 4 || (c >= 1);
        if (has) {
          const uint4 lo = (j < 4) ? D[c][u][0] : D[c > 0 ? c - 1 : 0][u][0];
          const uint4 hi = (j < 4) ? D[c][u][1] : D[c > 0 ? c - 1 : 0][u][1];
          const int db = 1 + 2 * ((j < 4) ? c : c - 1) + (j >> 2);
          const uint32_t rowb = stage + db * kDBlockBytes + r * 128;
          const uint32_t c0 = 2 * (j & 3);
          sts_v4(rowb + (((c0 + odd_first) ^ sw) << 4), odd_first ? hi : lo);
          sts_v4(rowb + (((c0 + 1 - odd_first) ^ sw) << 4), odd_first ? lo : hi);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.bar(kBarKvFull + 4 * st + c));
    }
  }
}

// Producers for bf16 rows (1024 bytes, no quantisation): the row's 16-byte
// piece q holds elements 8q .. 8q + 7, i.e. unit q % 8 of d-block q / 8.
// Thread (row_lo, j): rows row_lo and row_lo + 32, pieces 16c + j and
// 16c + 8 + j of chunk c (unit j of d-blocks 2c and 2c + 1), copied as they
// are. The loads of a tile are issued after the previous tile is stored.
__device__ void producer_role_bf16(const qsfm_params& p, const Smem& sm, int* fault) {
  const int ptid = threadIdx.x - kSoftThreads;  // 0..255 (8 producer warps)
  const int lane = threadIdx.x & 31;
  const int row_lo = ptid >> 3;  // 0..31
  const int j = ptid & 7;
  const int* rows = reinterpret_cast<const int*>(sm.ptr + kSRows);
  const int* kind = reinterpret_cast<const int*>(sm.ptr + kSRowKind);
  constexpr int kRow = QSFM_BF16_ROW_BYTES;

  int pr[2];
  uint4 R[4][2][2];  // [chunk][row][d-block of the chunk]

  auto fetch = [&](uint32_t n) -> bool {
    const uint32_t slot = n % kRing;
    if (!warp_wait_or_abort(sm, kBarRowsFull + slot, (n / kRing) & 1, fault)) return false;
    const int kd = kind[slot];
    pr[0] = rows[slot * kTileRows + row_lo];
    pr[1] = rows[slot * kTileRows + row_lo + 32];
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.bar(kBarRowsEmpty + slot));
    if (kd < 0) return false;
    const uint8_t* pool = static_cast<const uint8_t*>(kd ? p.cmp_kv : p.ori_kv);
    const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const bool v = pr[u] >= 0;
      const uint8_t* base = pool + size_t(v ? pr[u] : 0) * kRow + 16 * j;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        R[c][u][0] = v ? ldg_stream_v4(base + 256 * c) : z;
        R[c][u][1] = v ? ldg_stream_v4(base + 256 * c + 128) : z;
      }
    }
    return true;
  };

  for (uint32_t n = 0; fetch(n); ++n) {
    const uint32_t st = n & 1;
    if (!warp_wait_or_abort(sm, kBarKvEmpty + st, ((n >> 1) & 1) ^ 1, fault)) return;
    const uint32_t stage = sm.base + kSK + st * kStageBytes;
    if (j == 0) {
      int* valid = reinterpret_cast<int*>(sm.ptr + kSValid) + st * kTileRows;
      valid[row_lo] = pr[0] >= 0;
      valid[row_lo + 32] = pr[1] >= 0;
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int r = row_lo + 32 * u;
        const uint32_t unit = (uint32_t(j) ^ uint32_t(r & 7)) << 4;
        sts_v4(stage + (2 * c) * kDBlockBytes + r * 128 + unit, R[c][u][0]);
        sts_v4(stage + (2 * c + 1) * kDBlockBytes + r * 128 + unit, R[c][u][1]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.bar(kBarKvFull + 4 * st + c));
    }
  }
}

// ------------------------------------------------------------- MMA issue
// k-step s of d-block db: A (K~) at +db*8 KB + s*32 B, B (Q) at +db*8 KB + s*32 B.
template <int kDb, int kS>
__device__ __forceinline__ void qk_mma(uint32_t d, uint64_t a0, uint64_t b0) {
  constexpr uint32_t off = uint32_t((kDb * 8192 + kS * 32) >> 4);
  if constexpr ((kDb | kS) == 0)
    mma_bf16_at<off, off>(d, a0, b0, kIdescQK, 0u);
  else
    mma_bf16_acc_at<off, off>(d, a0, b0, kIdescQK);
}

// PV for head-dim chunk kC: A (V~^T, MN-major) at +kC*16 KB + ks*2 KB,
// B (P, MN-major) at +ks*2 KB.
template <int kC>
__device__ __forceinline__ void pv_chunk(uint32_t tmem, uint64_t a0, uint64_t b0, uint32_t acc0) {
  const uint32_t d = tmem + kTmemO + kC * 64;
  mma_bf16_at<uint32_t((kC * 16384 + 0 * 2048) >> 4), uint32_t((0 * 2048) >> 4)>(d, a0, b0, kIdescPV, acc0);
  mma_bf16_acc_at<uint32_t((kC * 16384 + 1 * 2048) >> 4), uint32_t((1 * 2048) >> 4)>(d, a0, b0, kIdescPV);
  mma_bf16_acc_at<uint32_t((kC * 16384 + 2 * 2048) >> 4), uint32_t((2 * 2048) >> 4)>(d, a0, b0, kIdescPV);
  mma_bf16_acc_at<uint32_t((kC * 16384 + 3 * 2048) >> 4), uint32_t((3 * 2048) >> 4)>(d, a0, b0, kIdescPV);
}

template <int kC>
__device__ __forceinline__ void qk_issue(uint32_t d, uint64_t a0, uint64_t b0) {
  qk_mma<2 * kC, 0>(d, a0, b0); qk_mma<2 * kC, 1>(d, a0, b0);
  qk_mma<2 * kC, 2>(d, a0, b0); qk_mma<2 * kC, 3>(d, a0, b0);
  qk_mma<2 * kC + 1, 0>(d, a0, b0); qk_mma<2 * kC + 1, 1>(d, a0, b0);
  qk_mma<2 * kC + 1, 2>(d, a0, b0); qk_mma<2 * kC + 1, 3>(d, a0, b0);
}

// Tile n of the CTA's sequence uses stage n & 1 (K~, S^T, P buffers); each
// barrier of a stage completes once per tile of that stage, so tile n waits
// for phase parity (n >> 1) & 1. Two threads issue tensor-core work, each
// blocking on its own inputs in program order: this one QK^T (and Q), the PV
// thread the PV products. QK^T(n) cannot run more than two tiles ahead of
// PV: its stage is refilled only after PV(n - 2) has completed.
__device__ void qk_role(const qsfm_params& p, const Smem& sm, Range rg, int T, uint32_t tmem,
                        const CUtensorMap* qmap, int* fault) {
  if ((threadIdx.x & 31) != 0) return;
  PieceIter pieces(&p, rg, T);
  TokenGeom g;
  auto next_live = [&](int& t_, int& lo_, int& hi_) {
    while (pieces.next(t_, g, lo_, hi_))
      if (lo_ < hi_) return true;
    return false;
  };
  auto load_q = [&](int t_) {
    mbar_arrive_expect_tx(sm.bar(kBarQFull), 64 * 1024);
#pragma unroll
    for (int db = 0; db < 8; ++db)
      tma_load_2d(sm.base + kSQ + db * 8192, qmap, db * 64, t_ * 64, sm.bar(kBarQFull));
  };
  int tok, lo, hi;
  bool have = next_live(tok, lo, hi);
  if (!have) return;
  load_q(tok);
  uint32_t n = 0, piece = 0;
  while (have) {
    int ntok = 0, nlo = 0, nhi = 0;
    const bool have_next = next_live(ntok, nlo, nhi);
    if (!wait_or_abort(sm, kBarQFull, piece & 1, fault)) return;
    for (int k = lo; k < hi; ++k, ++n) {
      const uint32_t st = n & 1, par = (n >> 1) & 1;
      // S^T buffer st is free once the softmax has read tile n - 2's scores
      if (!wait_or_abort(sm, kBarSFree + st, par ^ 1, fault)) return;
      const uint32_t d = tmem + kTmemS + 64 * st;
      const uint64_t a0 = make_sdesc_sw128(sm.base + kSK + st * kStageBytes, 16, 1024);
      const uint64_t b0 = make_sdesc_sw128(sm.base + kSQ, 16, 1024);
      if (!wait_or_abort(sm, kBarKvFull + 4 * st + 0, par, fault)) return;
      tc_fence_after();
      qk_issue<0>(d, a0, b0);
      if (!wait_or_abort(sm, kBarKvFull + 4 * st + 1, par, fault)) return;
      tc_fence_after();
      qk_issue<1>(d, a0, b0);
      if (!wait_or_abort(sm, kBarKvFull + 4 * st + 2, par, fault)) return;
      tc_fence_after();
      qk_issue<2>(d, a0, b0);
      if (!wait_or_abort(sm, kBarKvFull + 4 * st + 3, par, fault)) return;
      tc_fence_after();
      qk_issue<3>(d, a0, b0);
      mma_commit(sm.bar(kBarSFull + st));
      if (k == hi - 1 && have_next) {
        // Q of the next token once this token's last QK^T has read Q
        if (!wait_or_abort(sm, kBarSFull + st, par, fault)) return;
        load_q(ntok);
      }
    }
    ++piece;
    have = have_next;
    tok = ntok;
    lo = nlo;
    hi = nhi;
  }
}

__device__ void pv_role(const qsfm_params& p, const Smem& sm, Range rg, int T, uint32_t tmem,
                        int* fault) {
  if ((threadIdx.x & 31) != 0) return;
  PieceIter pieces(&p, rg, T);
  TokenGeom g;
  int tok, lo, hi;
  uint32_t n = 0, piece = 0;
  while (pieces.next(tok, g, lo, hi)) {
    if (lo >= hi) continue;
    for (int k = lo; k < hi; ++k, ++n) {
      const uint32_t st = n & 1;
      if (!wait_or_abort(sm, kBarPFull + st, (n >> 1) & 1, fault)) return;
      if (k == lo && piece > 0) {
        // the previous piece's epilogue must have read O^T before it is overwritten
        if (!wait_or_abort(sm, kBarOFree, (piece - 1) & 1, fault)) return;
      }
      tc_fence_after();
      const uint64_t a0 = make_sdesc_sw128(sm.base + kSK + st * kStageBytes, kDBlockBytes, 1024);
      const uint64_t b0 = make_sdesc_sw128(sm.base + kSP + st * kPBytes, 16, 1024);
      const uint32_t acc0 = k == lo ? 0u : 1u;
      pv_chunk<0>(tmem, a0, b0, acc0);
      pv_chunk<1>(tmem, a0, b0, acc0);
      pv_chunk<2>(tmem, a0, b0, acc0);
      pv_chunk<3>(tmem, a0, b0, acc0);
      mma_commit(sm.bar(kBarKvEmpty + st));  // stage (K~ and P) released
      if (k == hi - 1) mma_commit(sm.bar(kBarODone));
    }
    ++piece;
  }
}

// ------------------------------------------------------ softmax + epilogue
// Warp q reads the 16 tensor-memory lanes 32q..32q+15 of an S^T buffer, i.e.
// tile rows 16q..16q+15. In the accumulator-fragment layout thread l holds
// rows ra = 16q + l/4 and ra + 8, heads 8j + 2(l%4) + e (j = 0..7, e = 0, 1):
//   x[4j + 2r + e] = S^T[ra + 8r, 8j + 2(l%4) + e].
// Its 16 heads are indexed i = 2j + e in l[].
__device__ void softmax_role(const qsfm_params& p, const Smem& sm, Range rg, int T, uint32_t tmem,
                             const Workspace& ws, int c_idx, int* fault) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = tid;  // epilogue: head-dim element inside a 128-d chunk
  const int ra = 16 * warp + (lane >> 2);
  const int hq = 2 * (lane & 3);
  const uint32_t lane_base = uint32_t(32 * warp) << 16;
  const float qk_scale = p.softmax_scale * kLog2e;
  float* m_used = sm.f(kSMUsed);
  float* alpha = sm.f(kSAlpha);
  float* inv = sm.f(kSInv);
  float* red = sm.f(kSRed);
  PieceIter pieces(&p, rg, T);
  uint32_t n = 0, pieces_live = 0;
  int t, lo, hi;
  TokenGeom g;
  bool have = pieces.next(t, g, lo, hi);
  int n_tiles = g.n_tiles;
  while (have) {
    const bool whole = (lo == 0 && hi == n_tiles);
    // this thread's head sink (log2 units); the unit's heads start at unit_head0
    const float sink2 =
        (tid < 64 && p.sinks != nullptr) ? __ldg(p.sinks + unit_head0(p, t) + tid) * kLog2e : -INFINITY;
    const int slot = (t == rg.t0) ? 2 * c_idx : 2 * c_idx + 1;
    const bool writable = whole || slot < ws.slots;  // split pieces need the workspace
    if (!writable && tid == 0) atomicOr(fault, QSFM_FAULT_METADATA);
    float l[16], m[16];  // row sums and running max (log2 units) of this thread's 16 heads
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      l[i] = 0.f;
      m[i] = -INFINITY;
    }
    if (tid < 64) m_used[tid] = -INFINITY;
    named_sync(kBarSoft, kSoftThreads);
    for (int k = lo; k < hi; ++k, ++n) {
      const uint32_t st = n & 1, par = (n >> 1) & 1;
      // Lane 0 of each warp polls. After an abort the waits fall through at
      // once; the softmax warps keep running the same named-barrier sequence
      // so that none of them blocks.
      warp_wait_or_abort(sm, kBarKvFull + 4 * st, par, fault);
      const int* valid = reinterpret_cast<const int*>(sm.ptr + kSValid) + st * kTileRows;
      const bool va = valid[ra] != 0, vb = valid[ra + 8] != 0;
      warp_wait_or_abort(sm, kBarSFull + st, par, fault);
      tc_fence_after();
      const uint32_t s_addr = tmem + kTmemS + 64 * st + lane_base;
      float x[32];
      tmem_ld16x256b_x8(s_addr, x);
      tmem_ld_wait();
      bool move = true;  // the first tile of a piece always sets the max
      if (k != lo) {
        // Fast path: t = score * scale - m (log2 units), P = 2^t computed
        // before the vote; valid only if no t exceeds 8 anywhere in the tile.
        float tmax = -INFINITY;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int ia = 4 * (i >> 1) + (i & 1);
          const float ta = va ? fmaf(x[ia], qk_scale, -m[i]) : -INFINITY;
          const float tb = vb ? fmaf(x[ia + 2], qk_scale, -m[i]) : -INFINITY;
          tmax = fmaxf(tmax, fmaxf(ta, tb));
          x[ia] = ex2_approx(ta);
          x[ia + 2] = ex2_approx(tb);
        }
        move = named_sync_or(kBarSoft, kSoftThreads, tmax > kRescaleLog2);  // also true against -inf
        if (!move) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int ia = 4 * (i >> 1) + (i & 1);
            l[i] += x[ia] + x[ia + 2];
          }
        }
      }
      if (move) {
        // Slow path: the scores again (S^T buffer st is not reused before
        // this tile's PV has completed), then move the running max.
        if (k != lo) {
          tmem_ld16x256b_x8(s_addr, x);
          tmem_ld_wait();
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          x[4 * jj + 0] = va ? x[4 * jj + 0] * qk_scale : -INFINITY;
          x[4 * jj + 1] = va ? x[4 * jj + 1] * qk_scale : -INFINITY;
          x[4 * jj + 2] = vb ? x[4 * jj + 2] * qk_scale : -INFINITY;
          x[4 * jj + 3] = vb ? x[4 * jj + 3] * qk_scale : -INFINITY;
        }
        // tile max per head over the 64 rows
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          v[i] = fmaxf(x[4 * (i >> 1) + (i & 1)], x[4 * (i >> 1) + 2 + (i & 1)]);
        reduce_rows16<true>(v);  // lane l: heads 2l, 2l + 1
        red[warp * 64 + 2 * lane] = v[0];
        red[warp * 64 + 2 * lane + 1] = v[1];
        named_sync(kBarSoft, kSoftThreads);
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
        named_sync(kBarSoft, kSoftThreads);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int h = 8 * (i >> 1) + hq + (i & 1);
          l[i] *= alpha[h];
          m[i] = m_used[h];
        }
        if (k != lo) {
          // O^T at this thread's head-dim lane, all heads, once the PV product
          // of tile n - 1 has completed
          warp_wait_or_abort(sm, kBarKvEmpty + ((n - 1) & 1), ((n - 1) >> 1) & 1, fault);
          tc_fence_after();
#pragma unroll 1
          for (int q16 = 0; q16 < 16; ++q16) {
            float o[16];
            const uint32_t addr = tmem + kTmemO + 16 * q16 + lane_base;
            tmem_ld16(addr, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] *= alpha[16 * (q16 & 3) + i];
            tmem_st16(addr, o);
          }
          tmem_st_wait();
        }
        // P = 2^(x - m_used) and the row sums
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float mz = m[i] == -INFINITY ? 0.f : m[i];
          const int ia = 4 * (i >> 1) + (i & 1);
          x[ia] = ex2_approx(x[ia] - mz);
          x[ia + 2] = ex2_approx(x[ia + 2] - mz);
          l[i] += x[ia] + x[ia + 2];
        }
      }
      // the scores are no longer needed: the buffer can take tile n + 2
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.bar(kBarSFree + st));
      // P into its stage as [64 rows][64 heads] bf16 with the 128-B swizzle
      // (the MN-major B operand of PV)
      const uint32_t pbase = sm.base + kSP + st * kPBytes;
      const int mi = lane >> 3, jr = lane & 7;
      const uint32_t prow = pbase + uint32_t(16 * warp + 8 * (mi & 1) + jr) * 128;
#pragma unroll
      for (int gq = 0; gq < 4; ++gq) {
        const uint32_t hg = uint32_t(2 * gq + (mi >> 1));
        stmatrix_x4(prow + ((hg ^ uint32_t(jr)) << 4),
                    pack_bf16(x[8 * gq + 0], x[8 * gq + 1]), pack_bf16(x[8 * gq + 2], x[8 * gq + 3]),
                    pack_bf16(x[8 * gq + 4], x[8 * gq + 5]), pack_bf16(x[8 * gq + 6], x[8 * gq + 7]));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.bar(kBarPFull + st));
    }
    // The next piece's geometry, read now: its loads overlap the wait for
    // this piece's last PV product.
    int t_next = 0, lo_next = 0, hi_next = 0;
    const bool have_next = pieces.next(t_next, g, lo_next, hi_next);
    const int n_tiles_next = g.n_tiles;
    // ---------------- epilogue of the piece
    const bool any = lo < hi;
    if (any) {
      reduce_rows16<false>(l);  // lane l: heads 2l, 2l + 1 of this warp's rows
      red[warp * 64 + 2 * lane] = l[0];
      red[warp * 64 + 2 * lane + 1] = l[1];
    }
    named_sync(kBarSoft, kSoftThreads);
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
    named_sync(kBarSoft, kSoftThreads);
    if (any) {
      warp_wait_or_abort(sm, kBarODone, pieces_live & 1, fault);
      tc_fence_after();
    }
    // O^T in blocks of 128 d x 32 heads: lane = head-dim element, columns =
    // heads. Whole tokens go out through the P buffers, idle now: each block
    // is written there as 32 rows of 256 bytes ([head][d], bf16), then read
    // back 16 bytes per thread and stored with 16-byte stores (a warp writes
    // two 256-byte output rows per store); the two buffers alternate, so one
    // barrier per block suffices. Split pieces store fp32 rows directly (the
    // 32 lanes of a warp write 128 consecutive bytes per head).
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        const int h0 = 32 * half;
        const int blk = 2 * c + half;
        float o[32];
        if (any) {
          tmem_ld32(tmem + kTmemO + 64 * c + 32 * half + lane_base, o);
          tmem_ld_wait();
          // 1 / denominator per head, read into registers before any store
          // (the stores below could alias inv[] as far as the compiler knows)
          float iv[32];
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 v4 = *reinterpret_cast<const float4*>(inv + h0 + i);
            iv[i] = v4.x;
            iv[i + 1] = v4.y;
            iv[i + 2] = v4.z;
            iv[i + 3] = v4.w;
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= iv[i];
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0.f;
        }
        if (whole) {
          // every thread has read block blk - 2 back from this buffer before
          // the barrier of block blk - 1
          const uint32_t box = sm.base + kSP + uint32_t(blk & 1) * kPBytes;
#pragma unroll
          for (int i = 0; i < 32; ++i) sts_b16(box + uint32_t(i * 256 + 2 * row), __float2bfloat16_rn(o[i]));
          named_sync(kBarSoft, kSoftThreads);
          uint8_t* out = static_cast<uint8_t*>(p.attn_out) +
                         ((size_t(t) * 64 + h0) * kDim + 128 * c) * 2;
#pragma unroll
          for (int q = tid; q < 512; q += kSoftThreads) {  // q = 16-byte piece: head q / 16
            const uint32_t off = uint32_t(q >> 4) * 256 + uint32_t(q & 15) * 16;
            const uint4 v = lds_v4(box + off);
            *reinterpret_cast<uint4*>(out + size_t(q >> 4) * kDim * 2 + (q & 15) * 16) = v;
          }
        } else if (writable) {
          float* out = ws.out + (size_t(slot) * 64 + h0) * kDim + 128 * c + row;
#pragma unroll
          for (int i = 0; i < 32; ++i) out[size_t(i) * kDim] = o[i];
        }
      }
    }
    if (any) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.bar(kBarOFree));
      ++pieces_live;
    }
    named_sync(kBarSoft, kSoftThreads);  // m_used / inv / red are reused by the next piece
    if (*sm.abort_flag()) break;         // uniform: read after the barrier
    have = have_next;
    t = t_next;
    lo = lo_next;
    hi = hi_next;
    n_tiles = n_tiles_next;
  }
}

// Runs before the plan is readable, while the plan kernel still runs: warms
// L2 with the inputs of the token this CTA most likely starts with (the plan
// cuts equal-cost tokens evenly, so CTA c of G starts near token c T / G):
// its Q, its index list, its first two ori tiles and its first four cmp
// tiles. Only prefetches, so a wrong guess costs bandwidth, never results;
// each address is checked against its buffer first. Thread i of the
// producer warps takes ori slot i (i < 128) or cmp slot i - 128.
template <int kFmt>
__device__ __noinline__ void warm_first_token(const qsfm_params& p, int T, int c, int G, int i) {
  const int t = int((long long)c * T / G);
  if (t >= T) return;
  if (i == 0)
    bulk_prefetch_l2(static_cast<const uint8_t*>(p.q) + size_t(t) * kHeads * kDim * 2,
                     kHeads * kDim * 2);
  if (p.cmp_sparse_indices != nullptr && i < 32 && 32 * i < p.k2)
    prefetch_l2(p.cmp_sparse_indices + size_t(t >> unit_shift(p)) * p.k2 + 32 * i);
  const TokenGeom g = token_geom(p, t);
  int pos = -1;
  bool cmp = false;
  if (i < 2 * kTileRows) {
    if (i < g.n_ori) pos = g.ori_lo + i;
  } else {
    const int k = i - 2 * kTileRows;
    if (k < g.n_cmp) {
      cmp = true;
      pos = p.cmp_sparse_indices != nullptr ? __ldg(p.cmp_sparse_indices + size_t(g.tok) * p.k2 + k) : k;
      if (pos >= g.cmp_vis) pos = -1;
    }
  }
  if (pos < 0) return;
  const int col = pos / kBlock;
  const int width = cmp ? p.cmp_max_blocks : p.ori_max_blocks;
  if (col >= width) return;
  const int blk = __ldg((cmp ? p.cmp_block_table : p.ori_block_table) + size_t(g.b) * width + col);
  if (blk < 0 || blk >= (cmp ? p.cmp_num_blocks : p.ori_num_blocks)) return;
  const size_t row = size_t(blk) * kBlock + pos % kBlock;
  if constexpr (kFmt == QSFM_KV_PACKED640) {
    bulk_prefetch_l2(static_cast<const uint8_t*>(cmp ? p.cmp_kv : p.ori_kv) + row * QSFM_PACKED_ROW_BYTES,
                     QSFM_PACKED_ROW_BYTES);
  } else if constexpr (kFmt == QSFM_KV_BF16) {
    bulk_prefetch_l2(static_cast<const uint8_t*>(cmp ? p.cmp_kv : p.ori_kv) + row * QSFM_BF16_ROW_BYTES,
                     QSFM_BF16_ROW_BYTES);
  } else {
    bulk_prefetch_l2(static_cast<const uint8_t*>(cmp ? p.cmp_kv : p.ori_kv) + row * kDim, kDim);
    prefetch_l2((cmp ? p.cmp_scale : p.ori_scale) + row * kScales);
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
  if (warp >= kSoftWarps && warp < kSoftWarps + kProdWarps)
    warm_first_token<kFmt>(p, T, blockIdx.x, gridDim.x, tid - kSoftThreads);
  grid_dependency_wait();   // the plan (and every input) is written by now
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
    for (int i = 0; i < 4 * kStages; ++i) mbar_init(sm.bar(kBarKvFull + i), kProdWarps);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(sm.bar(kBarKvEmpty + i), 1);
      mbar_init(sm.bar(kBarSFull + i), 1);
      mbar_init(sm.bar(kBarSFree + i), kSoftWarps);
      mbar_init(sm.bar(kBarPFull + i), kSoftWarps);
    }
    mbar_init(sm.bar(kBarODone), 1);
    mbar_init(sm.bar(kBarOFree), kSoftWarps);
    for (int i = 0; i < kRing; ++i) {
      mbar_init(sm.bar(kBarRowsFull + i), 1);
      mbar_init(sm.bar(kBarRowsEmpty + i), kProdWarps);
    }
    *sm.abort_flag() = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(sm.tmem_slot(), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_slot();

  if (warp < kSoftWarps) {
    softmax_role(p, sm, rg, T, tmem, ws, c, fault);
  } else if (warp < kMmaWarp) {
    if constexpr (kFmt == QSFM_KV_PACKED640)
      producer_role_packed(p, sm, fault);
    else if constexpr (kFmt == QSFM_KV_BF16)
      producer_role_bf16(p, sm, fault);
    else
      producer_role(p, sm, fault);
  } else if (warp == kMmaWarp) {
    qk_role(p, sm, rg, T, tmem, &qmap, fault);
  } else if (warp == kPvWarp) {
    pv_role(p, sm, rg, T, tmem, fault);
  } else {
    resolver_role<kFmt>(p, sm, rg, T, fault);
  }

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
