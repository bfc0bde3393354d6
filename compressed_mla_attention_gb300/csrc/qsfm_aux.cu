// Planner, split-KV combine and debug-gather kernels (sm_103a).
//
// Planner: the split-core plan that QuantSparseFlashMlaMetadata produces for
// QuantSparseFlashMla (its function description: metadata is generated
// before the main op and passed to it; the metadata parameter row and the
// constraint "metadata ... shape fixed at [1024]"). Here it runs on the GPU
// from the device-resident lengths, so no host read-back is needed.
//
// Combine: merges the partial results of a token whose KV tiles were split
// over several CTAs, using the log-sum-exp of each part
// (torch_npu.npu_fused_infer_attention_score, output section, softmaxLse:
// lse exists so that attention split along S can be merged), and adds the
// per-head sink once (QuantSparseFlashMla parameter table row "sinks").
#include <cub/block/block_scan.cuh>
#include <cuda_runtime.h>

#include "qsfm_device.cuh"
#include "qsfm_internal.h"

namespace qsfm {
namespace {

constexpr int kPlanThreads = 1024;

__device__ __forceinline__ long long lmin(long long a, long long b) { return a < b ? a : b; }
__device__ __forceinline__ long long lmax(long long a, long long b) { return a > b ? a : b; }

// One CTA. Cost of a token = its KV tiles + 1 (loading Q, writing O). The
// total cost W is cut into G equal ranges. In split mode a cut may fall
// inside a token at a tile boundary; otherwise cuts snap to the start of the
// token that contains them.
__global__ void __launch_bounds__(kPlanThreads)
    plan_kernel(const qsfm_params p, const int T, const int g_max, const int split,
                int32_t* meta) {
  using Scan = cub::BlockScan<long long, kPlanThreads>;
  __shared__ typename Scan::TempStorage scan_tmp;
  __shared__ long long s_total[2];
  const int tid = threadIdx.x;
  // the attention kernel may take its place on the SMs now; it reads the
  // plan only after this grid has completed
  grid_launch_dependents();
  const int per = (T + kPlanThreads - 1) / kPlanThreads;
  const int ta = min(T, tid * per), tb = min(T, ta + per);
  // tiles per token, kept for the second pass for the first kKeep tokens
  // (beyond them they are recomputed)
  constexpr int kKeep = 6144;
  __shared__ int s_tiles[kKeep];
  long long cost = 0;
  for (int t = ta; t < tb; ++t) {
    const int n = token_geom(p, t).n_tiles;
    if (t < kKeep) s_tiles[t] = n;
    cost += n + 1;
  }
  long long pre, total;
  Scan(scan_tmp).ExclusiveSum(cost, pre, total);
  if (tid == 0) {
    s_total[0] = total;
    s_total[1] = total - T;  // every token costs its tiles + 1
  }
  __syncthreads();
  const long long W = s_total[0];
  int G;
  if (T == 0) G = 0;
  else if (split) G = int(lmin(g_max, lmax(1, s_total[1])));
  else G = min(g_max, T);

  if (tid == 0) {
    meta[0] = kMetaMagic;
    meta[1] = G;
    meta[2] = T;
    meta[3] = int(lmin(W, 0x7fffffffLL));
    meta[4] = split;
    meta[5] = int(lmin(s_total[1], 0x7fffffffLL));
    meta[6] = 0;
    meta[7] = 0;
    meta[kMetaHeader + 2 * G] = T;
    meta[kMetaHeader + 2 * G + 1] = 0;
  }
  if (G == 0) return;
  long long pos = pre;
  for (int t = ta; t < tb; ++t) {
    const int n = t < kKeep ? s_tiles[t] : token_geom(p, t).n_tiles;
    const long long ct = n + 1;
    // boundaries c with floor(c W / G) in [pos, pos + ct)
    long long c_lo = (pos * G + W - 1) / W;
    long long c_hi = ((pos + ct) * G + W - 1) / W - 1;
    c_lo = lmax(c_lo, 0);
    c_hi = lmin(c_hi, (long long)G - 1);
    for (long long cc = c_lo; cc <= c_hi; ++cc) {
      const long long target = cc * W / G;
      const long long o = target - pos;
      const int k = split ? int(lmax(0, lmin(o - 1, n > 0 ? n - 1 : 0))) : 0;
      meta[kMetaHeader + 2 * cc] = t;
      meta[kMetaHeader + 2 * cc + 1] = k;
    }
    pos += ct;
  }
}

// A fixed grid of blocks, each holding the plan's cuts in shared memory.
// Work item = (a token whose tiles were split over several CTAs, a head);
// the items are dealt to the warps of all blocks. The token is owned by its
// first cut that falls inside it; its parts are the ranges of that cut's
// predecessor and of the following cuts that start inside it. Lane l of a
// warp holds head-dim elements 4l..4l+3 of each 128-wide quarter, so each
// part's partial row is read with coalesced 512-byte loads.
constexpr int kCombineThreads = 256;
constexpr int kCombineBlocksPerCta = 4;
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const qsfm_params p, const int T, const Workspace ws, int* fault) {
  using Scan = cub::BlockScan<int, kCombineThreads>;
  __shared__ typename Scan::TempStorage scan_tmp;
  __shared__ int s_cut[2 * (QSFM_MAX_CTAS + 1)];
  __shared__ int s_owner[QSFM_MAX_CTAS];  // owning cut of the i-th split token
  __shared__ int s_nowned;
  grid_dependency_wait();  // the attention kernel's partial results
  const int32_t* meta = p.metadata;
  if (meta[0] != kMetaMagic || meta[2] != T) return;
  const int G = meta[1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // A plan made for more CTAs (or without split mode) than this call's
  // workspace holds would send the reads below past the workspace: refuse it.
  if (G < 0 || G > QSFM_MAX_CTAS || 2 * G > ws.slots || meta[4] != 1) {
    if (tid == 0 && blockIdx.x == 0) atomicOr(fault, QSFM_FAULT_METADATA);
    return;
  }
  for (int i = tid; i < 2 * (G + 1); i += kCombineThreads) s_cut[i] = meta[kMetaHeader + i];
  __syncthreads();
  // cut c (1 <= c < G) owns its token when it falls inside it and the
  // previous cut does not fall inside the same token
  int own = 0;
  if (tid >= 1 && tid < G) {
    const int t = s_cut[2 * tid], k = s_cut[2 * tid + 1];
    own = (k > 0 && t >= 0 && t < T && !(s_cut[2 * tid - 2] == t && s_cut[2 * tid - 1] > 0)) ? 1 : 0;
  }
  int pos, total;
  Scan(scan_tmp).ExclusiveSum(own, pos, total);
  if (own) s_owner[pos] = tid;
  if (tid == 0) s_nowned = total;
  __syncthreads();
  const int items = s_nowned * 64;
  const int warps_total = gridDim.x * (kCombineThreads / 32);
  for (int it = blockIdx.x * (kCombineThreads / 32) + warp; it < items; it += warps_total) {
    const int cb = s_owner[it >> 6], h = it & 63;
    const int t = s_cut[2 * cb];
    // the parts: ranges [cut c, cut c + 1) for c = cb - 1, cb, ... whose end
    // lies past the token's start (split-mode cuts never start past a
    // token's last tile, so every such range holds tiles of t)
    // in flight with the lse loads; t is a work unit (see unit_shift)
    const float sk = p.sinks != nullptr ? __ldg(p.sinks + unit_head0(p, t) + h) : -INFINITY;
    const int c_begin = cb - 1;
    int c_end = cb;
    while (c_end < G && s_cut[2 * c_end] <= t) ++c_end;
    const int m = c_end - c_begin;
    // lane i takes parts i, i + 32, ...: slot, lse
    auto part = [&](int i, int& sl, float& li) {
      const int c = c_begin + i;
      const int t1 = s_cut[2 * c + 2], k1 = s_cut[2 * c + 3];
      const bool ov = t1 > t || (t1 == t && k1 > 0);
      sl = (s_cut[2 * c] == t) ? 2 * c : 2 * c + 1;
      li = ov ? ws.lse[size_t(sl) * 64 + h] : -INFINITY;
    };
    float L = -INFINITY;
    for (int i0 = 0; i0 < m; i0 += 32) {
      int sl;
      float li = -INFINITY;
      if (i0 + lane < m) part(i0 + lane, sl, li);
      L = fmaxf(L, li);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) L = fmaxf(L, __shfl_xor_sync(0xffffffffu, L, o));
    float sum = 0.f;
    for (int i0 = 0; i0 < m && L > -INFINITY; i0 += 32) {
      int sl;
      float li = -INFINITY;
      if (i0 + lane < m) part(i0 + lane, sl, li);
      if (li > -INFINITY) sum += expf(li - L);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float lse_all = L > -INFINITY ? L + logf(sum) : -INFINITY;
    float denom_log = lse_all;
    if (p.sinks != nullptr && lse_all > -INFINITY) {
      const float mx = fmaxf(lse_all, sk);
      denom_log = mx + logf(expf(lse_all - mx) + expf(sk - mx));
    }
    if (p.return_lse && lane == 0) p.softmax_lse[size_t(t) * 64 + h] = lse_all;
    float4 acc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i0 = 0; i0 < m && lse_all > -INFINITY; i0 += 32) {
      // weights of this group of parts, one per lane, then broadcast
      int sl = 0;
      float li = -INFINITY;
      if (i0 + lane < m) part(i0 + lane, sl, li);
      const float w = li > -INFINITY ? expf(li - denom_log) : 0.f;
      const int mg = min(32, m - i0);
      for (int i = 0; i < mg; i += 4) {
        float4 v[4][4];
        float wi[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int src_lane = min(i + u, mg - 1);
          wi[u] = (i + u < mg) ? __shfl_sync(0xffffffffu, w, src_lane) : 0.f;
          const int su = __shfl_sync(0xffffffffu, sl, src_lane);
          const float* src = ws.out + (size_t(su) * 64 + h) * kDim + 4 * lane;
#pragma unroll
          for (int q = 0; q < 4; ++q) v[u][q] = __ldg(reinterpret_cast<const float4*>(src + 128 * q));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            acc[q].x += wi[u] * v[u][q].x;
            acc[q].y += wi[u] * v[u][q].y;
            acc[q].z += wi[u] * v[u][q].z;
            acc[q].w += wi[u] * v[u][q].w;
          }
      }
    }
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.attn_out) + (size_t(t) * 64 + h) * kDim + 4 * lane;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc[q].x, acc[q].y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc[q].z, acc[q].w);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(out + 128 * q) = pk;
    }
  }
}

// One CTA per requested token, one warp per tile: every tile is resolved by
// resolve_tile_rows with the lane mapping of the attention kernel's resolver
// warp (lane l: slots l, l + 32, l + 64, l + 96 of the tile), and each
// slot's logical row, and optionally its pool bytes, are written in the
// order the kernel visits them (ori window rows, then cmp slots), without
// the padding of partial tiles.
__global__ void __launch_bounds__(128)
    debug_gather_kernel(const qsfm_params p, const int T, const int32_t* tokens, int max_rows,
                        uint8_t* rows_out, float* scales_out, int32_t* row_ids_out,
                        int32_t* counts_out, int* fault) {
  const int i = blockIdx.x;
  const int t = tokens[i];
  if (t < 0 || t >= T) {
    if (threadIdx.x == 0) counts_out[i] = 0;
    return;
  }
  const TokenGeom g = token_geom(p, t << unit_shift(p));  // the token's first unit
  if (threadIdx.x == 0) counts_out[i] = g.n_ori + g.n_cmp;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int row_bytes = kv_row_bytes(p.kv_layout);
  for (int k = warp; k < g.n_tiles; k += blockDim.x >> 5) {
    const int ks[1] = {k};
    const bool live[1] = {true};
    int lgs[1][4], prs[1][4];
    bool cmps[1];
    resolve_tile_rows<1>(p, g, ks, live, lane, fault, lgs, prs, cmps);
    const bool cmp = cmps[0];
    const int* lg = lgs[0];
    const int* pr = prs[0];
    const uint8_t* pool = static_cast<const uint8_t*>(cmp ? p.cmp_kv : p.ori_kv);
    const float* spool = cmp ? p.cmp_scale : p.ori_scale;
    for (int u = 0; u < 4; ++u) {
      const int in_tile = (cmp ? (k - g.ori_tiles) : k) * kTileRows + lane + 32 * u;
      if (in_tile >= (cmp ? g.n_cmp : g.n_ori)) continue;  // padding of a partial tile
      const int s = cmp ? g.n_ori + in_tile : in_tile;
      if (s >= max_rows) continue;
      row_ids_out[size_t(i) * max_rows + s] = lg[u] >= 0 ? (int(cmp) << 30) | lg[u] : -1;
      if (rows_out == nullptr) continue;  // row ids only
      uint4* dst = reinterpret_cast<uint4*>(rows_out + (size_t(i) * max_rows + s) * row_bytes);
      const uint4* src = reinterpret_cast<const uint4*>(pool + size_t(pr[u] >= 0 ? pr[u] : 0) * row_bytes);
      for (int q = 0; q < row_bytes / 16; ++q) dst[q] = pr[u] >= 0 ? src[q] : make_uint4(0, 0, 0, 0);
      if (scales_out != nullptr) {
        float* dsc = scales_out + (size_t(i) * max_rows + s) * kScales;
        for (int q = 0; q < kScales; ++q) dsc[q] = pr[u] >= 0 ? spool[size_t(pr[u]) * kScales + q] : 0.f;
      }
    }
  }
}

}  // namespace

size_t workspace_bytes(int num_ctas) {
  const size_t slots = 2 * size_t(num_ctas);
  const size_t lse = (slots * 64 * sizeof(float) + 255) & ~size_t(255);
  return lse + slots * 64 * kDim * sizeof(float);
}

Workspace workspace_view(void* base, int num_ctas) {
  Workspace w;
  w.slots = 2 * num_ctas;
  const size_t lse = (size_t(w.slots) * 64 * sizeof(float) + 255) & ~size_t(255);
  w.lse = static_cast<float*>(base);
  w.out = reinterpret_cast<float*>(static_cast<uint8_t*>(base) + lse);
  return w;
}

// The bounded wait of the kernels against barriers nothing arrives on: the
// first wait runs out after timeout_ns and raises the abort flag, which ends
// the second (1000 times longer) wait early.
__global__ void bounded_wait_kernel(uint64_t timeout_ns, unsigned long long* elapsed, int* fault) {
  __shared__ uint64_t bars[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort = &abort_flag;
  const uint64_t t0 = globaltimer_ns();
  if (threadIdx.x == 0) {
    if (!mbar_wait_bounded(&bars[0], 0, abort, timeout_ns)) {
      *abort = 1;
      atomicOr(fault, QSFM_FAULT_TIMEOUT);
    }
    elapsed[0] = globaltimer_ns() - t0;
  } else if (threadIdx.x == 32) {
    mbar_wait_bounded(&bars[1], 0, abort, 1000 * timeout_ns);
    elapsed[1] = globaltimer_ns() - t0;
  }
}

cudaError_t launch_bounded_wait(uint64_t timeout_ns, unsigned long long* elapsed, int* fault,
                                cudaStream_t s) {
  bounded_wait_kernel<<<1, 64, 0, s>>>(timeout_ns, elapsed, fault);
  return cudaGetLastError();
}

cudaError_t launch_plan(const qsfm_params& p, int num_tokens, int num_ctas, int split,
                        int32_t* metadata, int* fault, cudaStream_t s) {
  (void)fault;
  plan_kernel<<<1, kPlanThreads, 0, s>>>(p, num_tokens, num_ctas, split, metadata);
  return cudaGetLastError();
}

cudaError_t launch_combine(const qsfm_params& p, int num_tokens, int num_ctas,
                           const Workspace& ws, int* fault, cudaStream_t s) {
  // Four blocks per planned CTA: every (split token, head) item of a full
  // decode batch gets a warp of its own, so the few dependent L2 round trips
  // of the items overlap instead of queueing in a warp.
  return launch_after_predecessor(combine_kernel, dim3(kCombineBlocksPerCta * num_ctas),
                                  dim3(kCombineThreads), 0, s, p, num_tokens, ws, fault);
}

cudaError_t launch_debug_gather(const qsfm_params& p, const int32_t* tokens, int n,
                                int max_rows, uint8_t* rows_out, float* scales_out,
                                int32_t* row_ids_out, int32_t* counts_out, int* fault,
                                cudaStream_t s) {
  const int T = p.layout_q == QSFM_LAYOUT_BSND ? p.batch * p.max_s1 : p.total_t;
  debug_gather_kernel<<<n, 128, 0, s>>>(p, T, tokens, max_rows, rows_out, scales_out,
                                        row_ids_out, counts_out, fault);
  return cudaGetLastError();
}

}  // namespace qsfm
