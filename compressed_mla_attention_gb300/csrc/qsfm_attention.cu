// Attention kernel of the quantized shared-KV sparse MLA forward (sm_103a).
//
// Computes, for every planned (token, KV-tile range) piece,
//   O = softmax([Q K~^T * softmax_scale, sink]) V~  with K~ = V~
// (QuantSparseFlashMla, function description formula; sink from its
// parameter table row "sinks"; lse from KvQuantSparseAttnSharedKv, parameter
// table row softmax_lse).
//
// Orientation. The contractions run transposed so that the KV-row dimension
// (128 rows per tile) is the MMA M dimension and the 64 heads are N:
//   S^T[j, h]  = sum_d K~[j, d] Q[h, d]      (M = 128 rows, N = 64, K = 512)
//   O^T[d, h] += sum_j V~[j, d] P[h, j]      (M = 128 d per chunk, N = 64,
//                                             K = 128 rows, 4 chunks)
// Both accumulators live in tensor memory: S^T in 64 columns, O^T in 256.
// One dequantised bf16 tile (128 rows x 512, 128-B swizzle, 8 d-blocks of
// 16 KB) is the K-major A operand of the first product and, read through an
// MN-major descriptor, the A operand of the second.
//
// Warp roles (13 warps; at most 4 per SM sub-partition, so 128 registers):
//   warps 0-3   softmax + epilogue. Thread i owns TMEM lane i: KV row i of the
//               tile for S^T (all 64 heads), head-dim element i of a 128-d
//               chunk for O^T.
//   warps 4-11  producers: resolve the paged rows of a tile, load their fp8
//               bytes and scales into registers one tile ahead, dequantise
//               them chunk by chunk (a chunk = 128 rows x 128 d = 2 d-blocks)
//               into the tile as soon as the previous tile's PV product has
//               released that chunk.
//   warp 12     tcgen05 issue (one thread): Q by TMA, QK^T per chunk as the
//               chunks arrive, PV per chunk, commits that release chunks.
// mbarriers carry every hand-off; every wait is bounded in time.
//
// Softmax: the running max m_used per head is moved only when a tile's max
// exceeds it by more than 8 (log2 units); a named-barrier vote detects that
// case, so most tiles need no cross-thread max reduction. When it moves, O^T
// and the per-thread sums l are rescaled exactly. P <= 2^8 in bf16.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "qsfm_device.cuh"
#include "qsfm_internal.h"

namespace qsfm {
namespace {

constexpr int kSoftWarps = 4;
constexpr int kProdWarps = 8;
constexpr int kMmaWarp = kSoftWarps + kProdWarps;
constexpr int kThreads = (kMmaWarp + 1) * 32;
constexpr int kSoftThreads = kSoftWarps * 32;
constexpr int kBarSoft = 1;  // named barrier id of the softmax warps

// shared memory map (byte offsets from a 1024-aligned base)
constexpr uint32_t kSK = 0;                      // K~: 8 d-blocks x 128 rows x 128 B
constexpr uint32_t kSQ = kSK + 8 * 128 * 128;    // Q: 8 d-blocks x 64 heads x 128 B
constexpr uint32_t kSP = kSQ + 8 * 64 * 128;     // P^T: 128 rows x 64 heads (bf16)
constexpr uint32_t kSRedMax = kSP + 128 * 128;   // [4][64] f32
constexpr uint32_t kSRedSum = kSRedMax + 1024;   // [2][4][64] f32 (per tile, double-buffered)
constexpr uint32_t kSLRun = kSRedSum + 2048;     // [64] f32 running sums
constexpr uint32_t kSMUsed = kSLRun + 256;       // [64] f32
constexpr uint32_t kSAlpha = kSMUsed + 256;      // [64] f32
constexpr uint32_t kSInv = kSAlpha + 256;        // [64] f32
constexpr uint32_t kSValid = kSInv + 256;        // [2][128] i32
constexpr uint32_t kSBar = kSValid + 1024;       // mbarriers, tmem base, flags
constexpr uint32_t kSmemBytes = kSBar + 256;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;

// mbarrier slots
constexpr int kBarQFull = 0;
constexpr int kBarKvFull = 1;   // 4 chunks
constexpr int kBarKvEmpty = 5;  // 4 chunks
constexpr int kBarSFull = 9;
constexpr int kBarPFull = 10;
constexpr int kBarODone = 11;
constexpr int kBarOFree = 12;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = 256;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kIdescQK = make_idesc_bf16(128, 64, /*a_mn=*/0, /*b_mn=*/0);
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

// Max (kMax) or sum over the 32 lanes of a warp of 32 values per lane.
// Afterwards lane l holds the result for value index l.
template <bool kMax>
__device__ __forceinline__ float warp_reduce32(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
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

struct Smem {
  uint32_t base;
  uint8_t* ptr;
  __device__ float* f(uint32_t off) const { return reinterpret_cast<float*>(ptr + off); }
  __device__ uint64_t* bar(int i) const { return reinterpret_cast<uint64_t*>(ptr + kSBar) + i; }
  __device__ uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(ptr + kSBar + 128); }
  __device__ volatile int* abort_flag() const {
    return reinterpret_cast<volatile int*>(ptr + kSBar + 136);
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

// ------------------------------------------------------------- producers
// One tile job: the physical row (block * 128 + offset, -1 = masked) of each
// of this thread's 4 rows, and which pool the tile reads (a tile never mixes
// ori and cmp rows).
struct JobRows {
  int prow[4];
  int cmp;
};

__device__ __forceinline__ void resolve_job(const qsfm_params& p, int tok, int k, const TokenGeom& g,
                                            int row_lo, int* fault, JobRows& jr) {
  jr.cmp = k >= g.ori_tiles;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const RowRef ref = resolve_slot(p, g, tok, k, row_lo + 32 * u, fault);
    const uint8_t* pool = static_cast<const uint8_t*>(jr.cmp ? p.cmp_kv : p.ori_kv);
    jr.prow[u] = ref.row >= 0 ? int((ref.kv - pool) / kDim) : -1;
  }
}

__device__ void producer_role(const qsfm_params& p, const Smem& sm, Range rg, int T, int* fault) {
  const int ptid = threadIdx.x - kSoftThreads;  // 0..255 (8 producer warps)
  const int lane = threadIdx.x & 31;
  const int row_lo = ptid >> 3;   // this thread's rows: row_lo + 32u, u = 0..3
  const int j = ptid & 7;         // its 16-byte slot inside each 128-byte chunk of a row
  const int odd_first = j >> 2;   // j >= 4 stores its odd 16-B chunk first (no bank conflicts)
  JobIter jobs(&p, rg, T);

  JobRows cur, nxt;
  float csc[4];  // scale j of each row (this lane's share of the row's 8 scales)
  uint4 R[4][4];  // fp8 bytes [chunk][row unit], loaded one tile ahead

  auto load_job = [&](const JobRows& jr) {
    const uint8_t* pool = static_cast<const uint8_t*>(jr.cmp ? p.cmp_kv : p.ori_kv);
    const float* spool = jr.cmp ? p.cmp_scale : p.ori_scale;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool v = jr.prow[u] >= 0;
      const uint8_t* src = pool + size_t(v ? jr.prow[u] : 0) * kDim + 16 * j;
#pragma unroll
      for (int c = 0; c < 4; ++c) R[c][u] = v ? ldg_stream_v4(src + 128 * c) : make_uint4(0, 0, 0, 0);
      csc[u] = v ? __ldg(spool + size_t(jr.prow[u]) * kScales + j) : 0.f;
    }
  };

  int tok, k;
  TokenGeom g;
  bool have_cur = jobs.next(tok, k, g);
  if (!have_cur) return;
  resolve_job(p, tok, k, g, row_lo, fault, cur);
  load_job(cur);
  bool have_nxt = jobs.next(tok, k, g);
  if (have_nxt) resolve_job(p, tok, k, g, row_lo, fault, nxt);

  // The next tile's rows are loaded only after this tile's last chunk has
  // been published: the proxy fence and the release of each chunk's arrive
  // wait for the thread's outstanding loads, so loads issued earlier would
  // serialise every chunk on a memory round trip. Issued here, they overlap
  // the softmax and PV product of the current tile instead.
  uint32_t ph = 1;  // kv_empty starts free
  uint32_t tiles = 0;
  while (have_cur) {
    int* valid = reinterpret_cast<int*>(sm.ptr + kSValid) + (tiles & 1) * 128;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (!warp_wait_or_abort(sm, kBarKvEmpty + c, ph, fault)) return;
      if (c == 0 && j == 0) {
#pragma unroll
        for (int u = 0; u < 4; ++u) valid[row_lo + 32 * u] = cur.prow[u] >= 0;
      }
      const int src_lane = (lane & ~7) | (2 * c + (j >> 2));
      const uint32_t blk = sm.base + kSK + (2 * c + (j >> 2)) * 16384;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float sc = __shfl_sync(0xffffffffu, csc[u], src_lane);
        uint4 lo, hi;
        dequant16(R[c][u], sc, lo, hi);
        const int r = row_lo + 32 * u;
        const uint32_t sw = uint32_t(r & 7);
        const uint32_t rowb = blk + r * 128;
        const uint32_t c0 = 2 * (j & 3);
        sts_v4(rowb + (((c0 + odd_first) ^ sw) << 4), odd_first ? hi : lo);
        sts_v4(rowb + (((c0 + 1 - odd_first) ^ sw) << 4), odd_first ? lo : hi);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.bar(kBarKvFull + c));
    }
    ph ^= 1;
    ++tiles;
    have_cur = have_nxt;
    if (have_cur) {
      cur = nxt;
      load_job(cur);
      have_nxt = jobs.next(tok, k, g);
      if (have_nxt) resolve_job(p, tok, k, g, row_lo, fault, nxt);
    }
  }
}

// ------------------------------------------------------------- MMA issue
// k-step s of d-block db: A (K~) at +db*16 KB + s*32 B, B (Q) at +db*8 KB + s*32 B.
template <int kDb, int kS>
__device__ __forceinline__ void qk_mma(uint32_t d, uint64_t a0, uint64_t b0) {
  mma_bf16_at<uint32_t((kDb * 16384 + kS * 32) >> 4), uint32_t((kDb * 8192 + kS * 32) >> 4)>(
      d, a0, b0, kIdescQK, (kDb | kS) != 0);
}

// QK^T over chunk kC (d-blocks 2kC, 2kC+1) once the producers publish it.
template <int kC>
__device__ __forceinline__ bool qk_chunk(const Smem& sm, uint32_t tmem, uint64_t a0, uint64_t b0,
                                         uint32_t par, int* fault) {
  if (!wait_or_abort(sm, kBarKvFull + kC, par, fault)) return false;
  tc_fence_after();
  const uint32_t d = tmem + kTmemS;
  qk_mma<2 * kC, 0>(d, a0, b0); qk_mma<2 * kC, 1>(d, a0, b0);
  qk_mma<2 * kC, 2>(d, a0, b0); qk_mma<2 * kC, 3>(d, a0, b0);
  qk_mma<2 * kC + 1, 0>(d, a0, b0); qk_mma<2 * kC + 1, 1>(d, a0, b0);
  qk_mma<2 * kC + 1, 2>(d, a0, b0); qk_mma<2 * kC + 1, 3>(d, a0, b0);
  return true;
}

// PV for head-dim chunk kC: A (V~^T, MN-major) at +kC*32 KB + ks*2 KB,
// B (P^T) at +ks*2 KB; then release the chunk to the producers.
template <int kC>
__device__ __forceinline__ void pv_chunk(const Smem& sm, uint32_t tmem, uint64_t a0, uint64_t b0,
                                         uint32_t acc0) {
  const uint32_t d = tmem + kTmemO + kC * 64;
  mma_bf16_at<uint32_t((kC * 32768 + 0 * 2048) >> 4), uint32_t((0 * 2048) >> 4)>(d, a0, b0, kIdescPV, acc0);
  mma_bf16_at<uint32_t((kC * 32768 + 1 * 2048) >> 4), uint32_t((1 * 2048) >> 4)>(d, a0, b0, kIdescPV, 1u);
  mma_bf16_at<uint32_t((kC * 32768 + 2 * 2048) >> 4), uint32_t((2 * 2048) >> 4)>(d, a0, b0, kIdescPV, 1u);
  mma_bf16_at<uint32_t((kC * 32768 + 3 * 2048) >> 4), uint32_t((3 * 2048) >> 4)>(d, a0, b0, kIdescPV, 1u);
  mma_bf16_at<uint32_t((kC * 32768 + 4 * 2048) >> 4), uint32_t((4 * 2048) >> 4)>(d, a0, b0, kIdescPV, 1u);
  mma_bf16_at<uint32_t((kC * 32768 + 5 * 2048) >> 4), uint32_t((5 * 2048) >> 4)>(d, a0, b0, kIdescPV, 1u);
  mma_bf16_at<uint32_t((kC * 32768 + 6 * 2048) >> 4), uint32_t((6 * 2048) >> 4)>(d, a0, b0, kIdescPV, 1u);
  mma_bf16_at<uint32_t((kC * 32768 + 7 * 2048) >> 4), uint32_t((7 * 2048) >> 4)>(d, a0, b0, kIdescPV, 1u);
  mma_commit(sm.bar(kBarKvEmpty + kC));
}

__device__ void mma_role(const qsfm_params& p, const Smem& sm, Range rg, int T, uint32_t tmem,
                         const CUtensorMap* qmap, int* fault) {
  if ((threadIdx.x & 31) != 0) return;
  PieceIter pieces(&p, rg, T);
  TokenGeom g;
  // the next piece that has tiles
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
  uint32_t tiles = 0, pieces_done = 0, ph_q = 0;
  while (have) {
    int ntok = 0, nlo = 0, nhi = 0;
    const bool have_next = next_live(ntok, nlo, nhi);
    if (!wait_or_abort(sm, kBarQFull, ph_q, fault)) return;
    ph_q ^= 1;
    for (int k = lo; k < hi; ++k) {
      const uint32_t par = tiles & 1;
      // Fully unrolled: descriptors are the base plus compile-time offsets
      // (32 B per k-step, 16 KB / 8 KB per d-block), so one thread issues an
      // MMA as fast as the pipe takes it.
      const uint64_t a0 = make_sdesc_sw128(sm.base + kSK, 16, 1024);
      const uint64_t b0 = make_sdesc_sw128(sm.base + kSQ, 16, 1024);
      if (!qk_chunk<0>(sm, tmem, a0, b0, par, fault)) return;
      if (!qk_chunk<1>(sm, tmem, a0, b0, par, fault)) return;
      if (!qk_chunk<2>(sm, tmem, a0, b0, par, fault)) return;
      if (!qk_chunk<3>(sm, tmem, a0, b0, par, fault)) return;
      mma_commit(sm.bar(kBarSFull));
      if (k == hi - 1 && have_next) {
        // Q of the next token as soon as this token's last QK^T has read Q
        if (!wait_or_abort(sm, kBarSFull, par, fault)) return;
        load_q(ntok);
      }
      if (!wait_or_abort(sm, kBarPFull, par, fault)) return;
      if (k == lo && pieces_done > 0) {
        // the previous token's epilogue must have read O^T before it is overwritten
        if (!wait_or_abort(sm, kBarOFree, (pieces_done - 1) & 1, fault)) return;
      }
      tc_fence_after();
      const uint64_t pa0 = make_sdesc_sw128(sm.base + kSK, 16384, 1024);
      const uint64_t pb0 = make_sdesc_sw128(sm.base + kSP, 16, 1024);
      const uint32_t acc0 = k == lo ? 0u : 1u;
      pv_chunk<0>(sm, tmem, pa0, pb0, acc0);
      pv_chunk<1>(sm, tmem, pa0, pb0, acc0);
      pv_chunk<2>(sm, tmem, pa0, pb0, acc0);
      pv_chunk<3>(sm, tmem, pa0, pb0, acc0);
      if (k == hi - 1) mma_commit(sm.bar(kBarODone));
      ++tiles;
    }
    ++pieces_done;
    have = have_next;
    tok = ntok;
    lo = nlo;
    hi = nhi;
  }
}

// ------------------------------------------------------ softmax + epilogue
// Thread i owns row i of the tile: its 64 scores are handled as two halves
// of 32 heads, read from TMEM again for each pass to keep registers low.
__device__ __forceinline__ void load_scores(uint32_t taddr, bool rv, float scale, float (&x)[32]) {
  tmem_ld32(taddr, x);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) x[i] = rv ? x[i] * scale : -INFINITY;
}

__device__ void softmax_role(const qsfm_params& p, const Smem& sm, Range rg, int T, uint32_t tmem,
                             const Workspace& ws, int c_idx, int* fault) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = tid;  // KV row of the tile / head-dim element inside a 128-d chunk
  const uint32_t lane_base = uint32_t(32 * warp) << 16;
  const float qk_scale = p.softmax_scale * kLog2e;
  float* m_used = sm.f(kSMUsed);
  float* alpha = sm.f(kSAlpha);
  float* inv = sm.f(kSInv);
  float* lrun = sm.f(kSLRun);
  float* red_max = sm.f(kSRedMax);
  float* red_sum = sm.f(kSRedSum);
  PieceIter pieces(&p, rg, T);
  uint32_t tiles = 0, pieces_live = 0;
  int t, lo, hi;
  TokenGeom g;
  while (pieces.next(t, g, lo, hi)) {
    const bool whole = (lo == 0 && hi == g.n_tiles);
    const int slot = (t == rg.t0) ? 2 * c_idx : 2 * c_idx + 1;
    const bool writable = whole || slot < ws.slots;  // split pieces need the workspace
    if (!writable && tid == 0) atomicOr(fault, QSFM_FAULT_METADATA);
    if (tid < 64) {
      m_used[tid] = -INFINITY;
      lrun[tid] = 0.f;
    }
    named_sync(kBarSoft, kSoftThreads);
    bool pend = false;  // red_sum of the previous tile not yet added to lrun
    for (int k = lo; k < hi; ++k) {
      const uint32_t par = tiles & 1;
      // Lane 0 of each warp polls. After an abort the waits fall through at
      // once; the softmax warps keep running the same named-barrier sequence
      // so that none of them blocks.
      warp_wait_or_abort(sm, kBarKvFull, par, fault);
      const bool rv = reinterpret_cast<int*>(sm.ptr + kSValid)[par * 128 + row] != 0;
      warp_wait_or_abort(sm, kBarSFull, par, fault);
      tc_fence_after();
      bool exceed = false;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        float x[32];
        load_scores(tmem + kTmemS + lane_base + 32 * half, rv, qk_scale, x);
#pragma unroll
        for (int i = 0; i < 32; ++i) exceed |= x[i] > m_used[32 * half + i] + kRescaleLog2;
      }
      const bool move = named_sync_or(kBarSoft, kSoftThreads, exceed);  // also true against -inf
      if (pend && tid < 64) {
        const float* rs = red_sum + (par ^ 1) * 256;
        lrun[tid] += (rs[tid] + rs[64 + tid]) + (rs[128 + tid] + rs[192 + tid]);
      }
      if (move) {
        // move the running max: tile max per head over the 128 rows
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          float x[32];
          load_scores(tmem + kTmemS + lane_base + 32 * half, rv, qk_scale, x);
          red_max[warp * 64 + 32 * half + lane] = warp_reduce32<true>(x);
        }
        named_sync(kBarSoft, kSoftThreads);
        if (tid < 64) {
          const float mt = fmaxf(fmaxf(red_max[tid], red_max[64 + tid]),
                                 fmaxf(red_max[128 + tid], red_max[192 + tid]));
          const float mu = m_used[tid];
          float a = 1.f;
          if (mt > -INFINITY && (mu == -INFINITY || mt > mu + kRescaleLog2)) {
            a = (mu == -INFINITY) ? 0.f : exp2f(mu - mt);
            m_used[tid] = mt;
          }
          alpha[tid] = a;
          lrun[tid] *= a;
        }
        named_sync(kBarSoft, kSoftThreads);
        if (k != lo) {
          // O^T at this thread's head-dim lane, all heads (the previous PV
          // product has completed: this tile's QK^T waited for it)
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
              float o[32];
              const uint32_t addr = tmem + kTmemO + 64 * c + 32 * half + lane_base;
              tmem_ld32(addr, o);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] *= alpha[32 * half + i];
              tmem_st16(addr, o);
              tmem_st16(addr + 16, o + 16);
            }
          }
          tmem_st_wait();
        }
      }
      // P = exp2(x - m_used) -> the P^T row line (64 heads, 128 B, swizzled),
      // and the per-head sums of this warp's 32 rows
      const uint32_t prow = sm.base + kSP + row * 128;
      const uint32_t sw = uint32_t(row & 7);
      float* rs = red_sum + par * 256 + warp * 64;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        float x[32];
        load_scores(tmem + kTmemS + lane_base + 32 * half, rv, qk_scale, x);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float mu = m_used[32 * half + i];
          x[i] = exp2f(x[i] - (mu == -INFINITY ? 0.f : mu));
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint4 v;
          v.x = pack_bf16(x[8 * cc + 0], x[8 * cc + 1]);
          v.y = pack_bf16(x[8 * cc + 2], x[8 * cc + 3]);
          v.z = pack_bf16(x[8 * cc + 4], x[8 * cc + 5]);
          v.w = pack_bf16(x[8 * cc + 6], x[8 * cc + 7]);
          sts_v4(prow + ((uint32_t(4 * half + cc) ^ sw) << 4), v);
        }
        rs[32 * half + lane] = warp_reduce32<false>(x);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.bar(kBarPFull));
      pend = true;
      ++tiles;
    }
    // ---------------- epilogue of the piece
    const bool any = lo < hi;
    named_sync(kBarSoft, kSoftThreads);
    if (tid < 64 && writable) {
      float lt = lrun[tid];
      if (pend) {
        const float* rs = red_sum + ((tiles - 1) & 1) * 256;
        lt += (rs[tid] + rs[64 + tid]) + (rs[128 + tid] + rs[192 + tid]);
      }
      const float mu = m_used[tid];
      const float lse2 = lt > 0.f ? mu + log2f(lt) : -INFINITY;
      if (whole) {
        float den = lt;
        if (p.sinks != nullptr && lt > 0.f) den += exp2f(__ldg(p.sinks + tid) * kLog2e - mu);
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
    // O^T chunk by chunk: lane = head-dim element, columns = heads. Whole
    // tokens go through the (now idle) P buffer as bf16 [64 heads][128 d] so
    // that every head's 256-byte run is written with 16-byte stores; split
    // pieces write fp32 partial rows straight to the workspace.
    uint8_t* stage = sm.ptr + kSP;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        float o[32];
        if (any) {
          tmem_ld32(tmem + kTmemO + 64 * c + 32 * half + lane_base, o);
          tmem_ld_wait();
        }
        const int h0 = 32 * half;
        if (whole) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            reinterpret_cast<__nv_bfloat16*>(stage)[(h0 + i) * 128 + row] =
                __float2bfloat16_rn(any ? o[i] * inv[h0 + i] : 0.f);
        } else if (writable) {
          float* out = ws.out + (size_t(slot) * 64 + h0) * kDim + 128 * c + row;
#pragma unroll
          for (int i = 0; i < 32; ++i) out[size_t(i) * kDim] = any ? o[i] * inv[h0 + i] : 0.f;
        }
      }
      if (whole) {
        named_sync(kBarSoft, kSoftThreads);
        // 64 heads x 256 B = 1024 16-byte pieces, 8 per thread
        uint8_t* gout = static_cast<uint8_t*>(p.attn_out) + size_t(t) * 64 * kDim * 2 + 256 * c;
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int piece = it * kSoftThreads + tid;
          const int h = piece >> 4, part = piece & 15;
          const uint4 v = *reinterpret_cast<const uint4*>(stage + h * 256 + part * 16);
          *reinterpret_cast<uint4*>(gout + size_t(h) * kDim * 2 + part * 16) = v;
        }
        named_sync(kBarSoft, kSoftThreads);
      }
    }
    if (any) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.bar(kBarOFree));
      ++pieces_live;
    }
    named_sync(kBarSoft, kSoftThreads);  // m_used / lrun / inv are reused by the next piece
    if (*sm.abort_flag()) break;         // uniform: read after the barrier
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    attention_kernel(const qsfm_params p, const int T, const Workspace ws, int* fault,
                     const __grid_constant__ CUtensorMap qmap) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  Smem sm;
  sm.base = (raw_addr + 1023u) & ~1023u;
  sm.ptr = smem_raw + (sm.base - raw_addr);

  const int tid = threadIdx.x, warp = tid >> 5;
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
    for (int i = 0; i < 4; ++i) {
      mbar_init(sm.bar(kBarKvFull + i), kProdWarps);
      mbar_init(sm.bar(kBarKvEmpty + i), 1);
    }
    mbar_init(sm.bar(kBarSFull), 1);
    mbar_init(sm.bar(kBarPFull), kSoftWarps);
    mbar_init(sm.bar(kBarODone), 1);
    mbar_init(sm.bar(kBarOFree), kSoftWarps);
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
    producer_role(p, sm, rg, T, fault);
  } else {
    mma_role(p, sm, rg, T, tmem, &qmap, fault);
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
  cudaError_t e = cudaFuncSetAttribute(attention_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
  if (e != cudaSuccess) return e;
  CUtensorMap qmap;
  e = make_q_map(p.q, num_tokens, &qmap);
  if (e != cudaSuccess) return e;
  attention_kernel<<<num_ctas, kThreads, kSmemAlloc, s>>>(p, num_tokens, ws, fault, qmap);
  return cudaGetLastError();
}

}  // namespace qsfm
