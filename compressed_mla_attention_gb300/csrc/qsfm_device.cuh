// Device-side building blocks shared by the qsfm kernels (sm_103a).
//
//  * token geometry: which ori rows and cmp slots a query token attends
//    (QuantSparseFlashMla, parameter table rows ori_mask_mode, cmp_mask_mode,
//    ori_win_left/right, cmp_residual_kv, cmp_topk_length; its constraints on
//    the cmp length and cmp_len * cmp_ratio + residual; positions aligned
//    bottom-right as a RightDownCausal mask is);
//  * paged row resolution through the block tables (QuantSparseFlashMla
//    constraints, PageAttention bullets);
//  * thin inline-PTX wrappers for mbarrier and tcgen05 (TMEM allocation,
//    MMA, commit, TMEM loads/stores, fences).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "qsfm.h"

namespace qsfm {

constexpr int kHeads = QSFM_NUM_HEADS;        // N1
constexpr int kDim = QSFM_HEAD_DIM;           // D
constexpr int kBlock = QSFM_BLOCK_SIZE;       // tokens per KV block
constexpr int kScales = QSFM_SCALES_PER_ROW;  // fp32 scales per row
constexpr int kTileRows = 128;                // KV rows per attention tile
constexpr int kMetaMagic = 0x51534D31;        // "QSM1"
constexpr int kMetaHeader = 8;
// metadata layout (int32[1024]):
//   [0] magic  [1] G (CTAs with work)  [2] T (query tokens)  [3] total cost
//   [4] split flag  [5] total tiles (clipped)  [6..7] reserved
//   [8 + 2c], [9 + 2c]  c = 0..G : (token, tile) where CTA c's range begins;
//   CTA c covers [begin_c, begin_{c+1}) in (token, tile) order.

// ---------------------------------------------------------------- geometry
struct TokenGeom {
  int b;          // batch of the token
  int s2;         // ori length S2 of the batch
  int tok;        // query token of the unit
  int ori_lo;     // first ori row of the mask range
  int ori_hi;     // last ori row of the mask range (ori picks must lie in it)
  int n_ori;      // ori slots: rows ori_lo .. ori_hi, or ori index entries scanned
  int n_cmp;      // cmp slots: CSA index entries scanned, HCA visible rows
  int cmp_vis;    // visible compressed rows V (CSA entries must be < V)
  int ori_base;   // non-paged KV: tensor row of the batch's ori row 0
  int cmp_base;   // non-paged KV: tensor row of the batch's cmp row 0
  int ori_tiles;  // ceil(n_ori / kTileRows)
  int n_tiles;    // ori tiles + ceil(n_cmp / kTileRows)
};

__device__ __forceinline__ int div_floor(int a, int b) {  // b > 0
  int q = a / b;
  return (a % b != 0 && a < 0) ? q - 1 : q;
}

// Work units: the 64-head groups of the query tokens (one per token for
// N1 = 64, two for N1 = 128; the pages' N1 is 64 or 128). Unit u is token
// u >> unit_shift, heads 64 (u & 1) .. + 63 for N1 = 128, and the flat head
// rows of q, attn_out and softmax_lse of the unit are 64 u .. 64 u + 63.
__device__ __forceinline__ int unit_shift(const qsfm_params& p) { return p.n1 == 128 ? 1 : 0; }
__device__ __forceinline__ int unit_head0(const qsfm_params& p, int u) {
  return p.n1 == 128 ? 64 * (u & 1) : 0;
}

// Batch, position in the batch's chunk and chunk length of query token t.
__device__ __forceinline__ void token_batch(const qsfm_params& p, int t, int& b, int& s,
                                            int& s1) {
  if (p.layout_q == QSFM_LAYOUT_BSND) {
    b = t / p.max_s1;
    s = t - b * p.max_s1;
    s1 = p.max_s1;
  } else {
    int lo = 0, hi = p.batch - 1;  // last b with cu[b] <= t
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (__ldg(p.cu_seqlens_q + mid) <= t) lo = mid; else hi = mid - 1;
    }
    b = lo;
    int c0 = __ldg(p.cu_seqlens_q + b);
    s = t - c0;
    s1 = __ldg(p.cu_seqlens_q + b + 1) - c0;
  }
}

// Not inlined: called once per token / tile, and every inlined copy would
// grow the instruction footprint of the hot loops around it.
// Geometry of work unit u (its token's rows; see unit_shift).
static __device__ __forceinline__ TokenGeom token_geom(const qsfm_params& p, int u) {
  TokenGeom g;
  const int t = u >> unit_shift(p);
  g.tok = t;
  int s, s1;
  token_batch(p, t, g.b, s, s1);
  // every per-batch / per-token length this token may need, loaded together
  // (one memory round trip instead of a chain of them). KV storage
  // (QuantSparseFlashMla constraints on layout_kv): S2 is seqused_ori_kv
  // (paged; BSND when given, else the S dimension) or the cu_seqlens_ori_kv
  // difference (TND); the cmp length defaults to floor(S2 / r) (paged), the
  // S dimension (BSND) or the cu_seqlens_cmp_kv difference (TND).
  const bool tnd_kv = p.layout_kv == QSFM_LAYOUT_KV_TND;
  const int used_ori = p.seqused_ori_kv != nullptr ? __ldg(p.seqused_ori_kv + g.b) : p.ori_kv_len;
  const int cu_o0 = tnd_kv ? __ldg(p.cu_seqlens_ori_kv + g.b) : 0;
  const int cu_o1 = tnd_kv ? __ldg(p.cu_seqlens_ori_kv + g.b + 1) : 0;
  const bool tnd_cmp = tnd_kv && p.cmp_kv != nullptr;
  const int cu_c0 = tnd_cmp ? __ldg(p.cu_seqlens_cmp_kv + g.b) : 0;
  const int cu_c1 = tnd_cmp ? __ldg(p.cu_seqlens_cmp_kv + g.b + 1) : 0;
  const int used_q = p.seqused_q != nullptr ? __ldg(p.seqused_q + g.b) : 0;
  const int used_cmp = p.seqused_cmp_kv != nullptr ? __ldg(p.seqused_cmp_kv + g.b) : 0;
  const int resid = p.cmp_residual_kv != nullptr ? __ldg(p.cmp_residual_kv + g.b) : 0;
  const int topk = p.cmp_topk_length != nullptr ? __ldg(p.cmp_topk_length + t) : 0;
  const int otopk = p.ori_topk_length != nullptr ? __ldg(p.ori_topk_length + t) : 0;
  g.s2 = tnd_kv ? cu_o1 - cu_o0 : used_ori;
  g.ori_base = tnd_kv ? cu_o0 : p.layout_kv == QSFM_LAYOUT_KV_BSND ? g.b * p.ori_kv_len : 0;
  g.cmp_base = tnd_kv ? cu_c0 : p.layout_kv == QSFM_LAYOUT_KV_BSND ? g.b * p.cmp_kv_len : 0;
  g.ori_lo = 0; g.ori_hi = -1; g.n_ori = 0; g.n_cmp = 0; g.cmp_vis = 0;
  bool live = !(p.seqused_q != nullptr && s >= used_q);
  if (live) {
    const int pos = g.s2 - s1 + s;  // bottom-right aligned position
    int lo, hi;
    if (p.ori_mask_mode == 0) {
      lo = 0; hi = g.s2 - 1;
    } else if (p.ori_mask_mode == 3) {
      lo = 0; hi = min(g.s2 - 1, pos);
    } else {
      lo = p.ori_win_left < 0 ? 0 : max(0, pos - p.ori_win_left);
      hi = p.ori_win_right < 0 ? g.s2 - 1 : min(g.s2 - 1, pos + p.ori_win_right);
    }
    g.ori_lo = lo;
    g.ori_hi = hi;
    if (p.ori_sparse_indices != nullptr)  // discrete picks: slots = index entries scanned
      g.n_ori = p.ori_topk_length != nullptr ? max(0, min(p.k1, otopk)) : p.k1;
    else
      g.n_ori = max(0, hi - lo + 1);
    if (p.cmp_kv != nullptr) {
      const int r = p.cmp_ratio;
      const int cmp_len = p.seqused_cmp_kv ? used_cmp
                          : tnd_kv          ? cu_c1 - cu_c0
                          : p.layout_kv == QSFM_LAYOUT_KV_BSND ? p.cmp_kv_len
                                                               : g.s2 / r;
      const int res = resid;
      const int pc = cmp_len * r + res - s1 + s;
      g.cmp_vis = p.cmp_mask_mode == 3 ? max(0, min(cmp_len, div_floor(pc + 1, r))) : cmp_len;
      if (p.cmp_sparse_indices != nullptr) {
        g.n_cmp = p.k2;
        if (p.cmp_topk_length) g.n_cmp = max(0, min(p.k2, topk));
      } else {
        g.n_cmp = g.cmp_vis;
      }
    }
  }
  g.ori_tiles = (g.n_ori + kTileRows - 1) / kTileRows;
  g.n_tiles = g.ori_tiles + (g.n_cmp + kTileRows - 1) / kTileRows;
  return g;
}

// Rows of the four slots i0, i0 + 32, i0 + 64, i0 + 96 of tiles k[t] of unit
// g, for kN tiles t at once (0 <= i0 < 32): the one row resolution of the
// library. The attention kernel's resolver warp and the debug gather (one
// tile per call) call it with lane = i0, so the debug export shows exactly
// the rows the kernel reads.
//   logical[t][u]: the logical row of the slot in its KV sequence, -1 when
//               the slot is past the token's rows, a -1 / out-of-range
//               ori or cmp pick, or a row that could not be resolved;
//   prow[t][u]: the row's index in the KV tensor (paged: block * 128 +
//               offset; BSND: b * S + row; TND: cu_seqlens_*_kv[b] + row),
//               -1 when logical is -1;
//   cmp[t]:     false for ori tiles, true for cmp tiles.
// Tiles with live[t] false are skipped (all -1). A table column past the
// table width, a block id outside the pool or a non-paged row past the end
// of its tensor sets a fault bit (when fault is not null) and masks the
// slot: it is never read. The index loads of all slots are in flight
// together, then all their block-table loads.
template <int kN>
__device__ __forceinline__ void resolve_tile_rows(const qsfm_params& p, const TokenGeom& g,
                                                  const int (&k)[kN], const bool (&live)[kN], int i0,
                                                  int* fault, int (&logical)[kN][4],
                                                  int (&prow)[kN][4], bool (&cmp)[kN]) {
  int row[kN][4];
  bool ok[kN][4];
  const int32_t* cidx = p.cmp_sparse_indices + (size_t)g.tok * p.k2;
  const int32_t* oidx = p.ori_sparse_indices + (size_t)g.tok * p.k1;
#pragma unroll
  for (int t = 0; t < kN; ++t) {
    const bool ori = k[t] < g.ori_tiles;
    cmp[t] = !ori;
    const int base = (ori ? k[t] : k[t] - g.ori_tiles) * kTileRows + i0;
    const int n = ori ? g.n_ori : g.n_cmp;
    const bool picks = ori ? p.ori_sparse_indices != nullptr : p.cmp_sparse_indices != nullptr;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int slot = base + 32 * u;
      ok[t][u] = live[t] && slot < n;
      row[t][u] = ori ? g.ori_lo + slot : slot;
      if (picks && ok[t][u]) row[t][u] = __ldg((ori ? oidx : cidx) + slot);
    }
  }
  const bool paged = p.layout_kv == QSFM_LAYOUT_KV_PA_BBND;
  int blk[kN][4];
#pragma unroll
  for (int t = 0; t < kN; ++t) {
    const bool ori = !cmp[t];
    const int32_t* table = ori ? p.ori_block_table : p.cmp_block_table;
    const int width = ori ? p.ori_max_blocks : p.cmp_max_blocks;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      // picks count only inside the token's range: ori picks in its ori mask
      // range, cmp picks below the visible count (-1 never passes)
      if (ori && p.ori_sparse_indices != nullptr)
        ok[t][u] = ok[t][u] && row[t][u] >= g.ori_lo && row[t][u] <= g.ori_hi;
      if (!ori && p.cmp_sparse_indices != nullptr)
        ok[t][u] = ok[t][u] && row[t][u] >= 0 && row[t][u] < g.cmp_vis;
      const int col = ok[t][u] ? row[t][u] / kBlock : 0;
      if (paged && ok[t][u] && col >= width) {
        if (fault != nullptr) atomicOr(fault, ori ? QSFM_FAULT_ORI_TABLE_COL : QSFM_FAULT_CMP_TABLE_COL);
        ok[t][u] = false;
      }
      blk[t][u] = (paged && ok[t][u]) ? __ldg(table + (size_t)g.b * width + col) : 0;
    }
  }
#pragma unroll
  for (int t = 0; t < kN; ++t) {
    const bool ori = !cmp[t];
    if (paged) {
      const int nblocks = ori ? p.ori_num_blocks : p.cmp_num_blocks;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (ok[t][u] && (blk[t][u] < 0 || blk[t][u] >= nblocks)) {
          if (fault != nullptr) atomicOr(fault, ori ? QSFM_FAULT_ORI_BLOCK_ID : QSFM_FAULT_CMP_BLOCK_ID);
          ok[t][u] = false;
        }
        logical[t][u] = ok[t][u] ? row[t][u] : -1;
        prow[t][u] = ok[t][u] ? blk[t][u] * kBlock + row[t][u] % kBlock : -1;
      }
    } else {
      // BSND / TND KV: the batch's rows start at its base row; a row past
      // the end of the tensor (lengths larger than the tensor) is skipped
      const int rbase = ori ? g.ori_base : g.cmp_base;
      const int len = ori ? p.ori_kv_len : p.cmp_kv_len;
      const int lim = p.layout_kv == QSFM_LAYOUT_KV_TND ? len - rbase : len;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (ok[t][u] && row[t][u] >= lim) {
          if (fault != nullptr) atomicOr(fault, QSFM_FAULT_KV_ROW);
          ok[t][u] = false;
        }
        logical[t][u] = ok[t][u] ? row[t][u] : -1;
        prow[t][u] = ok[t][u] ? rbase + row[t][u] : -1;
      }
    }
  }
}

// Bytes of one KV row in the pool of each row format.
__host__ __device__ constexpr int kv_row_bytes(int fmt) {
  return fmt == QSFM_KV_PACKED640 ? QSFM_PACKED_ROW_BYTES : fmt == QSFM_KV_BF16 ? QSFM_BF16_ROW_BYTES : kDim;
}

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Wait until the barrier's phase with the given parity has completed.
// Bounded: returns false after `max_iters` polls (the caller reports a
// timeout instead of spinning forever).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t max_iters) {
  const uint32_t addr = smem_u32(bar);
  for (uint32_t it = 0; it < max_iters; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// One poll of a barrier phase: true once the phase with `parity` completed.
__device__ __forceinline__ bool mbar_test(uint32_t addr, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(addr), "r"(parity)
      : "memory");
  return done != 0;
}

// Non-blocking test of a barrier phase (for a thread that polls several).
__device__ __forceinline__ bool mbar_ready(uint32_t addr, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(addr), "r"(parity)
      : "memory");
  return done != 0;
}

// Hint: bring `bytes` bytes at `ptr` into L2 (ptr 16-byte aligned, bytes a
// multiple of 16); nothing is written to shared memory.
__device__ __forceinline__ void bulk_prefetch_l2(const void* ptr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(bytes) : "memory");
}

// Hint: bring the 128-byte line holding `ptr` into L2.
__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

// Wait for a barrier phase, bounded in time: gives up (returns false) after
// `timeout_ns` or as soon as *abort becomes non-zero. try_wait suspends the
// thread in hardware until the phase completes or a short time limit passes,
// so the loop polls rarely; only long waits back off further with sleeps.
// The polling loop is out of line, so each call site adds one test and a
// call: the many waits of a kernel then share one copy of the loop.
static __device__ __forceinline__ bool mbar_wait_poll(uint32_t addr, uint32_t parity, volatile int* abort,
                                            uint64_t timeout_ns) {
  const uint64_t start = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (it > 256) __nanosleep(64);
    if (mbar_test(addr, parity)) return true;
    if ((it & 15u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - start > timeout_ns) return false;
    }
  }
}

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort, uint64_t timeout_ns) {
  const uint32_t addr = smem_u32(bar);
  if (mbar_test(addr, parity)) return true;
  return mbar_wait_poll(addr, parity, abort, timeout_ns);
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Arrive and add `bytes` to the barrier's expected transaction count.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// 2-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Programmatic dependent launch: a kernel launched right after another one
// on the same stream with the programmatic-serialization attribute may start
// before its predecessor has finished; grid_dependency_wait() blocks until
// every grid it depends on has completed and its writes are visible (a no-op
// without such a dependency). grid_launch_dependents() lets the kernel that
// follows start its own prologue early.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier over `count` threads.
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier over `count` threads that also returns whether any of them
// passed pred = true.
__device__ __forceinline__ bool named_sync_or(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(uint32_t(pred)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Whole-warp TMEM allocation; the base address is written to *dst (smem).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (bf16 in, fp32 acc).
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One MMA with descriptors a_base + kAOff, b_base + kBOff, accumulating when
// `accumulate` != 0. The offsets (16-byte units, compile-time immediates)
// only move the 14-bit start-address field in the low word (the whole
// shared-memory window is below 256 KB), so a 32-bit add on the low word
// gives the same descriptor as a 64-bit add, in fewer instructions on the
// single issuing thread.
template <uint32_t kAOff, uint32_t kBOff>
__device__ __forceinline__ void mma_f16_at(uint32_t d_tmem, uint64_t a_base, uint64_t b_base, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .b32 alo, ahi, blo, bhi;\n .reg .b64 a, b;\n"
      " mov.b64 {alo, ahi}, %1;\n mov.b64 {blo, bhi}, %2;\n"
      " add.u32 alo, alo, %5;\n add.u32 blo, blo, %6;\n"
      " mov.b64 a, {alo, ahi};\n mov.b64 b, {blo, bhi};\n"
      " setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_base), "l"(b_base), "r"(idesc), "r"(accumulate), "n"(kAOff), "n"(kBOff)
      : "memory");
}

// Arrive on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32, A/B bf16 (or
// both f16 with f16 = true), M x N, each operand K-major (0) or MN-major (1).
__host__ __device__ constexpr uint32_t make_idesc_bf16(int m, int n, int a_mn, int b_mn, bool f16 = false) {
  return (1u << 4)                          // D format: f32
         | (f16 ? 0u : (1u << 7))           // A format: f16 (0) or bf16 (1)
         | (f16 ? 0u : (1u << 10))          // B format: f16 (0) or bf16 (1)
         | (uint32_t(a_mn) << 15)           // A major
         | (uint32_t(b_mn) << 16)           // B major
         | (uint32_t(n >> 3) << 17)         // N / 8
         | (uint32_t(m >> 4) << 24);        // M / 16
}

// Shared-memory matrix descriptor, 128-byte swizzle. Addresses are byte
// offsets in the CTA's shared window; lbo / sbo are byte strides.
__device__ __forceinline__ uint64_t make_sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFFu);
  d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
  d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
  d |= uint64_t(1) << 46;  // descriptor version for tcgen05
  d |= uint64_t(2) << 61;  // layout: SWIZZLE_128B
  return d;
}

// 32 lanes x 32 bit, 16 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])));
}

// 32 lanes x 32 bit, 32 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31])));
}

// 16 lanes x 256 bit, 8 repetitions along the columns (64 columns). Thread t
// of the warp receives, for repetition j, the accumulator-fragment quad
//   v[4j+0] = (lane t/4,     column 8j + 2(t%4)),  v[4j+1] = its column + 1,
//   v[4j+2] = (lane t/4 + 8, column 8j + 2(t%4)),  v[4j+3] = its column + 1,
// lanes counted from the warp's base lane in `taddr`.
__device__ __forceinline__ void tmem_ld16x256b_x8(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Four 8x8 b16 matrices to shared memory; thread t gives the address of row
// t%8 of matrix t/8 and, in register i, the pair (row t/4, columns 2(t%4),
// 2(t%4)+1) of matrix i.
__device__ __forceinline__ void stmatrix_x4(uint32_t saddr, uint32_t r0, uint32_t r1, uint32_t r2,
                                            uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(saddr),
               "r"(r0), "r"(r1), "r"(r2), "r"(r3)
               : "memory");
}

// 2^x by the hardware approximation (relative error about 2^-22; subnormal
// results flush to zero, 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ----------------------------------------------------------- fp8 dequant
// 2 e4m3fn values (low byte first) times `scale`, rounded to a bf16 pair.
__device__ __forceinline__ uint32_t dequant2(uint16_t two, float scale) {
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(two, __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
  __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
  return *reinterpret_cast<uint32_t*>(&b);
}

// The same with both products of a pair in one packed fp32 multiply
// (mul.rn.f32x2: each lane rounds like mul.rn.f32, subnormals kept), so the
// result is bit-identical to dequant2.
__device__ __forceinline__ uint32_t dequant2_x2(uint16_t two, uint64_t scale2) {
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(two, __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
  const uint64_t in = (uint64_t(__float_as_uint(f.y)) << 32) | __float_as_uint(f.x);
  uint64_t out;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(out) : "l"(in), "l"(scale2));
  __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(uint32_t(out)), __uint_as_float(uint32_t(out >> 32)));
  return *reinterpret_cast<uint32_t*>(&b);
}

// 16 fp8 bytes -> 16 bf16 (two 16-byte chunks), packed multiplies.
__device__ __forceinline__ void dequant16_x2(const uint4& in, float scale, uint4& lo, uint4& hi) {
  const uint64_t s2 = (uint64_t(__float_as_uint(scale)) << 32) | __float_as_uint(scale);
  lo.x = dequant2_x2(uint16_t(in.x & 0xFFFF), s2);
  lo.y = dequant2_x2(uint16_t(in.x >> 16), s2);
  lo.z = dequant2_x2(uint16_t(in.y & 0xFFFF), s2);
  lo.w = dequant2_x2(uint16_t(in.y >> 16), s2);
  hi.x = dequant2_x2(uint16_t(in.z & 0xFFFF), s2);
  hi.y = dequant2_x2(uint16_t(in.z >> 16), s2);
  hi.z = dequant2_x2(uint16_t(in.w & 0xFFFF), s2);
  hi.w = dequant2_x2(uint16_t(in.w >> 16), s2);
}

// 2 e4m3fn values (low byte first) -> f16x2 (exact), times the f16x2 scale
// pair s2 (one f16 multiply per lane, rounded once).
__device__ __forceinline__ uint32_t dequant2_f16(uint16_t two, uint32_t s2) {
  uint32_t h, r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(two));
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(s2));
  return r;
}

// 16 fp8 bytes -> 16 f16 (two 16-byte chunks) with the scale pair s2.
__device__ __forceinline__ void dequant16_f16(const uint4& in, uint32_t s2, uint4& lo, uint4& hi) {
  lo.x = dequant2_f16(uint16_t(in.x & 0xFFFF), s2);
  lo.y = dequant2_f16(uint16_t(in.x >> 16), s2);
  lo.z = dequant2_f16(uint16_t(in.y & 0xFFFF), s2);
  lo.w = dequant2_f16(uint16_t(in.y >> 16), s2);
  hi.x = dequant2_f16(uint16_t(in.z & 0xFFFF), s2);
  hi.y = dequant2_f16(uint16_t(in.z >> 16), s2);
  hi.z = dequant2_f16(uint16_t(in.w & 0xFFFF), s2);
  hi.w = dequant2_f16(uint16_t(in.w >> 16), s2);
}

// Two fp32 values rounded to an f16x2 pair (a in the low half).
__device__ __forceinline__ uint32_t pack_f16(float a, float b) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

// 16 fp8 bytes -> 16 bf16 (two 16-byte chunks).
__device__ __forceinline__ void dequant16(const uint4& in, float scale, uint4& lo, uint4& hi) {
  lo.x = dequant2(uint16_t(in.x & 0xFFFF), scale);
  lo.y = dequant2(uint16_t(in.x >> 16), scale);
  lo.z = dequant2(uint16_t(in.y & 0xFFFF), scale);
  lo.w = dequant2(uint16_t(in.y >> 16), scale);
  hi.x = dequant2(uint16_t(in.z & 0xFFFF), scale);
  hi.y = dequant2(uint16_t(in.z >> 16), scale);
  hi.z = dequant2(uint16_t(in.w & 0xFFFF), scale);
  hi.w = dequant2(uint16_t(in.w >> 16), scale);
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
  return v;
}

// Streaming read of data used once: no L1 allocation (the L1 left beside a
// large shared-memory carve-out is small).
__device__ __forceinline__ uint4 ldg_stream_v4(const void* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
  return v;
}

// 4-byte read when pred is true, else 0. Predicated (not a load and a
// select), so nothing waits for the load until its value is used.
__device__ __forceinline__ uint32_t ldg_pred_u32(const void* ptr, bool pred) {
  uint32_t v = 0;
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %2, 0;\n @p ld.global.nc.b32 %0, [%1];\n}"
               : "+r"(v)
               : "l"(ptr), "r"(uint32_t(pred)));
  return v;
}

// Streaming read of 8 bytes (8-byte aligned).
__device__ __forceinline__ uint2 ldg_stream_v2(const void* ptr) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(ptr));
  return v;
}

__device__ __forceinline__ void sts_b16(uint32_t saddr, __nv_bfloat16 v) {
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(saddr), "h"(*reinterpret_cast<const uint16_t*>(&v))
               : "memory");
}

__device__ __forceinline__ uint4 lds_v4(uint32_t saddr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(saddr)
               : "memory");
  return v;
}

__device__ __forceinline__ void sts_v4(uint32_t saddr, const uint4& v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(saddr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

}  // namespace qsfm
