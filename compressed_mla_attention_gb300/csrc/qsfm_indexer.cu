// Lightning-indexer top-k (QuantLightningIndexerV2, quant mode 1) for sm_103a.
//
// For every query token: score_j = sum_h W[h] ReLU(Sq[h] Sk[j] (Q[h] . K[j]))
// over the keys it may see, then the topk keys of largest score
// (QuantLightningIndexerV2, "功能说明": the formula and its three steps).
//
// One CTA per SM, persistent over query tokens. Per token:
//   * Q (heads x 128 e4m3 bytes) is copied by the threads into shared
//     memory with the 128-byte swizzle, zero rows up to N = heads rounded up
//     to 16 (the MMA's N);
//   * the keys stream in 128-row tiles, one paged block per tile: one TMA
//     box (128 rows x 128 bytes, 128-byte swizzle) plus a 512-byte bulk copy
//     of the block's key scales, four stages deep;
//   * S^T[j, h] = sum_d K[j, d] Q[h, d] on the tensor cores: tcgen05.mma
//     kind::f8f6f4 (e4m3 x e4m3, fp32 accumulate), M = 128 keys, N, K = 32 per
//     MMA, 4 MMAs per tile, into one of two TMEM accumulators;
//   * 8 epilogue warps read S^T (warp w: TMEM lane quarter w mod 4, heads
//     32 (w / 4 mod 2) .. + 31), each thread one key row, and reduce its heads
//     to a partial score; two partials per key make its score, kept in
//     shared memory (up to 32768 keys: 128 KB);
//   * all 320 threads then select the topk: a 4-pass radix select on the
//     scores' order-preserving 32-bit keys finds the k-th largest score,
//     and a block-wide scan writes the selected keys in ascending order
//     (equal scores: smaller key first), then -1.
// Roles: warp 0 TMA producer, warp 1 MMA issue, warps 2-9 epilogue; every
// mbarrier wait is bounded (timeout -> fault bit, abort flag, orderly exit).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "qsfm_device.cuh"

namespace qsfm {
namespace {

constexpr int kIxThreads = 320;
constexpr int kIxWarps = kIxThreads / 32;
constexpr int kIxDim = 128;        // bytes (= e4m3 elements) per query / key row
constexpr int kIxTile = 128;       // keys per tile (one paged block)
constexpr int kIxStages = 4;
constexpr int kIxMaxKeys = 32768;  // keys per token kept in shared memory
constexpr int kIxMaxHeads = 64;
constexpr int kIxBarEpi = 1;       // named barrier of the 8 epilogue warps
constexpr int kIxEpiThreads = 256;
constexpr uint64_t kIxTimeoutNs = 2000000000ull;

// shared memory map (byte offsets from a 1024-aligned base)
constexpr uint32_t kXKey = 0;                                      // [stage] 16 KB key tiles
constexpr uint32_t kXQ = kXKey + kIxStages * kIxTile * kIxDim;       // 64 rows x 128 B
constexpr uint32_t kXKs = kXQ + kIxMaxHeads * kIxDim;              // [stage][128] f32 key scales
constexpr uint32_t kXScore = kXKs + kIxStages * kIxTile * 4;       // [32768] f32 scores
constexpr uint32_t kXPart = kXScore + kIxMaxKeys * 4;              // [2 acc][2 half][128] f32
constexpr uint32_t kXW = kXPart + 2 * 2 * kIxTile * 4;             // [64] f32 weights
constexpr uint32_t kXSq = kXW + 256;                               // [64] f32 query scales
constexpr uint32_t kXHist = kXSq + 256;                            // [256] i32
constexpr uint32_t kXScan = kXHist + 1024;                         // [64] i32 scan scratch
constexpr uint32_t kXValid = kXScan + 256;                         // [stage] i32 tile valid
constexpr uint32_t kXBar = kXValid + 64;                           // barriers, tmem slot, flags
constexpr uint32_t kXBytes = kXBar + 256;
constexpr uint32_t kXAlloc = kXBytes + 1024;
static_assert(kXAlloc <= 232448, "indexer shared memory");

// barriers: full[4], empty[4], tfull[2], tempty[2]
constexpr int kXbFull = 0, kXbEmpty = 4, kXbTFull = 8, kXbTEmpty = 10, kXbDrain = 12, kXbCount = 13;
static_assert(kXbCount * 8 <= 128, "barriers overlap the tmem slot");

struct IxSmem {
  uint32_t base;
  uint8_t* ptr;
  __device__ uint64_t* bar(int i) const { return reinterpret_cast<uint64_t*>(ptr + kXBar) + i; }
  __device__ uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(ptr + kXBar + 128); }
  __device__ volatile int* abort_flag() const { return reinterpret_cast<volatile int*>(ptr + kXBar + 136); }
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

// 1-D bulk copy global -> shared, completing on `bar` (both addresses and
// the size multiples of 16 bytes).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mma_f8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// Batch, position and chunk length of query token t, and the keys it may
// see (0 for a padded row).
__device__ __forceinline__ void ix_token(const qsfm_indexer_params& p, int t, int& b, int& s, int& nvis) {
  int s1;
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
  const int sk = __ldg(p.seqused_k + b);
  if (p.seqused_q != nullptr && s >= __ldg(p.seqused_q + b)) {
    nvis = 0;
    return;
  }
  if (p.mask_mode == 0) {
    nvis = sk;
  } else {
    const int r = p.cmp_ratio;
    const int res = p.cmp_residual_k != nullptr ? __ldg(p.cmp_residual_k + b) : 0;
    const int pc = sk * r + res - s1 + s;
    nvis = max(0, min(sk, div_floor(pc + 1, r)));
  }
}

// Order-preserving 32-bit key of a score (-0 taken as +0).
__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f == 0.f ? 0.f : f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum of v over the block's 320 threads (scratch: 16 ints).
__device__ __forceinline__ int block_exclusive_scan(int v, int tid, int* scratch, int& total) {
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
    int w = lane < kIxWarps ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += u;
    }
    if (lane < kIxWarps) scratch[16 + lane] = w;
  }
  __syncthreads();
  total = scratch[16 + kIxWarps - 1];
  const int r = (warp ? scratch[16 + warp - 1] : 0) + incl - v;
  __syncthreads();  // scratch is reused by the next call
  return r;
}


// Top-k of the scores 0 .. n - 1 in shared memory into out[0 .. k): the keys
// of the k largest scores (the smaller key first among equal ones) in
// ascending key order, then -1; vals (bf16, or null) get the scores, -inf
// after them. Every thread of the block calls it.
__device__ void ix_select(const IxSmem& sm, int n, int k, int tid, int32_t* out, __nv_bfloat16* vals) {
  const float* sc = sm.f(kXScore);
  int* hist = sm.i(kXHist);
  int* scratch = sm.i(kXScan);
  const bool all = n <= k;
  uint32_t thr = 0;
  int need = 0;
  if (!all) {
    // radix select of the k-th largest key, 8 bits a pass from the top
    uint32_t prefix = 0, mask = 0;
    int remaining = k;  // of the keys matching the prefix, the rank wanted
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = tid; i < 256; i += kIxThreads) hist[i] = 0;
      __syncthreads();
      for (int j = tid; j < n; j += kIxThreads) {
        const uint32_t u = score_key(sc[j]);
        if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1);
      }
      __syncthreads();
      if (tid < 32) {
        // lane l holds bins 255 - 8l .. 248 - 8l, the largest first
        int c[8], sum = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          c[q] = hist[255 - 8 * tid - q];
          sum += c[q];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int u = __shfl_up_sync(0xffffffffu, incl, o);
          if (tid >= o) incl += u;
        }
        const int excl = incl - sum;
        if (excl < remaining && remaining <= incl) {  // exactly one lane
          int acc = excl;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (acc + c[q] >= remaining) {
              scratch[48] = 255 - 8 * tid - q;
              scratch[49] = acc;  // keys of larger bins
              break;
            }
            acc += c[q];
          }
        }
      }
      __syncthreads();
      prefix |= uint32_t(scratch[48]) << shift;
      mask |= 0xFFu << shift;
      remaining -= scratch[49];
      __syncthreads();
    }
    thr = prefix;      // the k-th largest key
    need = remaining;  // keys equal to it that are taken, smallest first
  }
  // ascending key order: thread tid owns keys j0 .. j1 - 1
  const int per = (n + kIxThreads - 1) / kIxThreads;
  const int j0 = min(n, tid * per), j1 = min(n, j0 + per);
  int eq = 0, gt = 0;
  if (!all)
    for (int j = j0; j < j1; ++j) {
      const uint32_t u = score_key(sc[j]);
      eq += u == thr;
      gt += u > thr;
    }
  int tot = 0;
  const int eq_rank0 = all ? 0 : block_exclusive_scan(eq, tid, scratch, tot);
  const int mine = all ? j1 - j0 : gt + max(0, min(eq, need - eq_rank0));
  int nsel = 0;
  int pos = block_exclusive_scan(mine, tid, scratch, nsel);
  int er = eq_rank0;
  for (int j = j0; j < j1; ++j) {
    bool take = all;
    if (!all) {
      const uint32_t u = score_key(sc[j]);
      take = u > thr || (u == thr && er < need);
      er += u == thr;
    }
    if (take) {
      out[pos] = j;
      if (vals != nullptr) vals[pos] = __float2bfloat16_rn(sc[j]);
      ++pos;
    }
  }
  for (int i = nsel + tid; i < k; i += kIxThreads) {
    out[i] = -1;
    if (vals != nullptr) vals[i] = __float2bfloat16_rn(-INFINITY);
  }
}


__global__ void __launch_bounds__(kIxThreads, 1)
    indexer_kernel(const qsfm_indexer_params p, const int T, int* fault, const __grid_constant__ CUtensorMap kmap) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  IxSmem sm;
  sm.base = (raw + 1023u) & ~1023u;
  sm.ptr = smem_raw + (sm.base - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int heads = p.heads;
  const int npad = max(16, (heads + 15) & ~15);  // the MMA's N
  if (tid == 0) {
    for (int i = 0; i < kIxStages; ++i) {
      mbar_init(sm.bar(kXbFull + i), 1);
      mbar_init(sm.bar(kXbEmpty + i), 1 + 8);  // the MMAs' commit and the 8 epilogue warps
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(sm.bar(kXbTFull + i), 1);
      mbar_init(sm.bar(kXbTEmpty + i), 8);
    }
    mbar_init(sm.bar(kXbDrain), 1);
    *sm.abort_flag() = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(sm.tmem_slot(), 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_slot();
  // e4m3 x e4m3 (format code 0 for A and B), fp32 accumulate, both K-major
  const uint32_t idesc = make_idesc_bf16(128, npad, 0, 0, true);
  float* wsm = sm.f(kXW);
  float* sqm = sm.f(kXSq);
  float* part = sm.f(kXPart);
  float* score = sm.f(kXScore);
  const float* ksm = sm.f(kXKs);
  int* valid = sm.i(kXValid);
  const uint8_t* q8 = static_cast<const uint8_t*>(p.query);
  uint32_t ctr = 0;  // tiles before this token (stage and phase of every barrier)
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    int b, s, nvis;
    ix_token(p, t, b, s, nvis);
    if (nvis > kIxMaxKeys) {
      if (tid == 0) atomicOr(fault, QSFM_FAULT_KV_ROW);
      nvis = kIxMaxKeys;
    }
    const int ntiles = (nvis + kIxTile - 1) / kIxTile;
    // the token's Q (rows >= heads zero), weights and query scales
    for (int i = tid; i < npad * 8; i += kIxThreads) {
      const int row = i >> 3, c = i & 7;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (row < heads) v = ldg_nc_v4(q8 + (size_t(t) * heads + row) * kIxDim + 16 * c);
      sts_v4(sm.base + kXQ + row * kIxDim + ((uint32_t(c) ^ uint32_t(row & 7)) << 4), v);
    }
    for (int i = tid; i < heads; i += kIxThreads) {
      wsm[i] = __ldg(p.weights + size_t(t) * heads + i);
      sqm[i] = __ldg(p.query_scale + size_t(t) * heads + i);
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (warp == 0) {
      if (lane == 0) {
        // producer: one paged block of keys and its scales per tile
        for (int i = 0; i < ntiles; ++i) {
          const uint32_t n = ctr + i, st = n % kIxStages;
          if (n >= kIxStages && !ix_wait(sm, kXbEmpty + st, ((n / kIxStages) & 1) ^ 1, fault)) break;
          int blk = -1;
          if (i < p.max_blocks) blk = __ldg(p.block_table + size_t(b) * p.max_blocks + i);
          else atomicOr(fault, QSFM_FAULT_CMP_TABLE_COL);
          if (blk < 0 || blk >= p.num_blocks) {
            if (i < p.max_blocks) atomicOr(fault, QSFM_FAULT_CMP_BLOCK_ID);
            valid[st] = 0;  // the tile's scores become -inf; nothing is read
            mbar_arrive(sm.bar(kXbFull + st));
          } else {
            valid[st] = 1;
            mbar_arrive_expect_tx(sm.bar(kXbFull + st), kIxTile * kIxDim + kIxTile * 4);
            tma_load_2d(sm.base + kXKey + st * (kIxTile * kIxDim), &kmap, 0, blk * kIxTile,
                        sm.bar(kXbFull + st));
            bulk_g2s(sm.base + kXKs + st * (kIxTile * 4), p.key_scale + size_t(blk) * kIxTile, kIxTile * 4,
                     sm.bar(kXbFull + st));
          }
        }
      }
    } else if (warp == 1) {
      if (lane == 0) {
        const uint64_t bdesc = make_sdesc_sw128(sm.base + kXQ, 16, 1024);
        for (int i = 0; i < ntiles; ++i) {
          const uint32_t n = ctr + i, st = n % kIxStages, a = n & 1;
          if (!ix_wait(sm, kXbFull + st, (n / kIxStages) & 1, fault)) break;
          if (n >= 2 && !ix_wait(sm, kXbTEmpty + a, ((n >> 1) & 1) ^ 1, fault)) break;
          tc_fence_after();
          const uint64_t adesc = make_sdesc_sw128(sm.base + kXKey + st * (kIxTile * kIxDim), 16, 1024);
          const uint32_t d = tmem + a * 64;
#pragma unroll
          for (int k = 0; k < kIxDim / 32; ++k)  // 32 e4m3 (32 bytes) of d per MMA
            mma_f8(d, adesc + uint64_t((k * 32) >> 4), bdesc + uint64_t((k * 32) >> 4), idesc, k > 0 ? 1u : 0u);
          mma_commit(sm.bar(kXbTFull + a));
          mma_commit(sm.bar(kXbEmpty + st));
        }
      }
    } else {
      // epilogue: warp w reads TMEM lanes 32 (w mod 4) .. + 31 (its key rows)
      // and heads 32 half .. + 31
      const int quarter = warp & 3, half = (warp - 2) >> 2;
      const int row = 32 * quarter + lane;
      // After a timeout the waits fail at once; the warps keep running the
      // same named-barrier sequence (no work) so that none of them blocks.
      bool alive = !*sm.abort_flag();
      for (int i = 0; i < ntiles; ++i) {
        const uint32_t n = ctr + i, st = n % kIxStages, a = n & 1;
        if (alive) alive = ix_warp_wait(sm, kXbTFull + a, (n >> 1) & 1, fault);
        if (alive) alive = ix_warp_wait(sm, kXbFull + st, (n / kIxStages) & 1, fault);  // the scales landed
        float acc = 0.f;
        int ok = 0;
        if (alive) {
          tc_fence_after();
          float x[32];
          const bool mine = half * 32 < heads;
          if (mine) {
            tmem_ld32(tmem + a * 64 + half * 32 + (uint32_t(32 * quarter) << 16), x);
            tmem_ld_wait();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(sm.bar(kXbTEmpty + a));
          const float sk = ksm[st * kIxTile + row];
          ok = valid[st];
          __syncwarp();
          if (lane == 0) mbar_arrive(sm.bar(kXbEmpty + st));  // the stage may be refilled
          if (mine) {
#pragma unroll
            for (int h = 0; h < 32; ++h) {
              const int hh = half * 32 + h;
              if (hh < heads) acc += wsm[hh] * fmaxf(0.f, (sqm[hh] * sk) * x[h]);
            }
          }
        }
        part[(a * 2 + half) * kIxTile + row] = acc;
        named_sync(kIxBarEpi, kIxEpiThreads);
        if (half == 0 && alive) {
          const int j = i * kIxTile + row;
          if (j < nvis) score[j] = ok ? part[(a * 2) * kIxTile + row] + part[(a * 2 + 1) * kIxTile + row] : -INFINITY;
        }
      }
    }
    __syncthreads();  // the token's scores are complete
    ctr += ntiles;
    if (*sm.abort_flag()) break;
    __nv_bfloat16* vals = p.return_value ? static_cast<__nv_bfloat16*>(p.sparse_values) + size_t(t) * p.topk : nullptr;
    ix_select(sm, nvis, p.topk, tid, p.sparse_indices + size_t(t) * p.topk, vals);
    __syncthreads();  // scores and scratch are reused by the next token
  }
  if (warp == 1 && lane == 0) {
    // every MMA issued above completes before tensor memory is freed
    mma_commit(sm.bar(kXbDrain));
    ix_wait(sm, kXbDrain, 0, fault);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// Tensor map of the key pool viewed as [num_blocks * 128 rows, 128 bytes],
// boxes of one block (128 x 128 bytes) with the 128-byte swizzle of the
// MMA's K-major operand.
cudaError_t make_key_map(const void* key, int num_blocks, CUtensorMap* map) {
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
  if (encode == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cuuint64_t(kIxDim), cuuint64_t(num_blocks) * kIxTile};
  const cuuint64_t strides[1] = {cuuint64_t(kIxDim)};
  const cuuint32_t box[2] = {kIxDim, kIxTile};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(key), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_indexer(const qsfm_indexer_params& p, int T, int* fault, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(indexer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kXAlloc);
  if (e != cudaSuccess) return e;
  CUtensorMap kmap;
  e = make_key_map(p.key, p.num_blocks, &kmap);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int grid = T < sms ? T : sms;
  indexer_kernel<<<grid, kIxThreads, kXAlloc, s>>>(p, T, fault, kmap);
  return cudaGetLastError();
}

}  // namespace qsfm
