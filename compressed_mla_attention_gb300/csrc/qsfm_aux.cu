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

struct Pair {
  int t, k;
};
__device__ __forceinline__ bool pair_less(Pair a, Pair b) {
  return a.t < b.t || (a.t == b.t && a.k < b.k);
}

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

// One CTA per cut: the CTA of the first cut that falls inside a token merges
// all parts of that token.
__global__ void __launch_bounds__(256)
    combine_kernel(const qsfm_params p, const int T, const Workspace ws, int* fault) {
  const int32_t* meta = p.metadata;
  if (meta[0] != kMetaMagic || meta[2] != T) return;
  const int G = meta[1];
  if (G < 0 || G > int(gridDim.x) || G > QSFM_MAX_CTAS) return;
  const int cb = blockIdx.x;
  if (cb < 1 || cb >= G) return;
  const Pair here{meta[kMetaHeader + 2 * cb], meta[kMetaHeader + 2 * cb + 1]};
  if (here.k <= 0 || here.t < 0 || here.t >= T) return;
  const Pair prev{meta[kMetaHeader + 2 * cb - 2], meta[kMetaHeader + 2 * cb - 1]};
  if (prev.t == here.t && prev.k > 0) return;  // an earlier cut owns this token
  const int t = here.t;
  const int n = token_geom(p, t).n_tiles;
  const Pair tok_lo{t, 0}, tok_hi{t, n};

  __shared__ int s_slot[QSFM_MAX_CTAS + 1];
  __shared__ float s_lse[64];    // log-sum-exp over all parts (sink excluded)
  __shared__ float s_denom[64];  // log of the full denominator (sink included)
  __shared__ int s_n;
  const int tid = threadIdx.x;
  if (tid == 0) {
    int m = 0;
    for (int c = cb - 1; c < G; ++c) {
      const Pair b0{meta[kMetaHeader + 2 * c], meta[kMetaHeader + 2 * c + 1]};
      if (b0.t > t) break;
      const Pair b1{meta[kMetaHeader + 2 * c + 2], meta[kMetaHeader + 2 * c + 3]};
      const Pair lo = pair_less(b0, tok_lo) ? tok_lo : b0;
      const Pair hi = pair_less(b1, tok_hi) ? b1 : tok_hi;
      if (pair_less(lo, hi)) s_slot[m++] = (b0.t == t) ? 2 * c : 2 * c + 1;
    }
    s_n = m;
  }
  __syncthreads();
  const int m = s_n;
  if (tid < 64) {
    float L = -INFINITY;
    for (int i = 0; i < m; ++i) L = fmaxf(L, ws.lse[size_t(s_slot[i]) * 64 + tid]);
    float lse_all = -INFINITY;
    if (L > -INFINITY) {
      float sum = 0.f;
      for (int i = 0; i < m; ++i) sum += expf(ws.lse[size_t(s_slot[i]) * 64 + tid] - L);
      lse_all = L + logf(sum);
    }
    float denom_log = lse_all;
    if (p.sinks != nullptr && lse_all > -INFINITY) {
      const float sk = __ldg(p.sinks + tid);
      const float mx = fmaxf(lse_all, sk);
      denom_log = mx + logf(expf(lse_all - mx) + expf(sk - mx));
    }
    s_lse[tid] = lse_all;
    s_denom[tid] = denom_log;
  }
  __syncthreads();
  if (p.return_lse && tid < 64) p.softmax_lse[size_t(t) * 64 + tid] = s_lse[tid];
  // 64 heads x 512 outputs; thread -> (head, 128-wide d range)
  const int h = tid >> 2, d0 = (tid & 3) * 128;
  const bool live = s_lse[h] > -INFINITY;
  const float dl = s_denom[h];
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.attn_out) + (size_t(t) * 64 + h) * kDim + d0;
  for (int d = 0; d < 128; d += 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 0; i < m && live; ++i) {
      const float li = ws.lse[size_t(s_slot[i]) * 64 + h];
      if (li == -INFINITY) continue;
      const float w = expf(li - dl);
      const float4 v = *reinterpret_cast<const float4*>(
          ws.out + (size_t(s_slot[i]) * 64 + h) * kDim + d0 + d);
      acc.x += w * v.x; acc.y += w * v.y; acc.z += w * v.z; acc.w += w * v.w;
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(out + d) = pk;
  }
}

// One CTA per requested token: writes the token's row slots in the order the
// attention kernel visits them (ori window rows, then cmp slots), without the
// padding of partial tiles.
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
  const TokenGeom g = token_geom(p, t);
  const int n_slots = g.n_ori + g.n_cmp;
  if (threadIdx.x == 0) counts_out[i] = n_slots;
  const int lim = min(n_slots, max_rows);
  for (int s = threadIdx.x; s < lim; s += blockDim.x) {
    int k, r;
    if (s < g.n_ori) {
      k = s / kTileRows;
      r = s % kTileRows;
    } else {
      const int cs = s - g.n_ori;
      k = g.ori_tiles + cs / kTileRows;
      r = cs % kTileRows;
    }
    const RowRef ref = resolve_slot(p, g, t, k, r, fault);
    uint4* dst = reinterpret_cast<uint4*>(rows_out + (size_t(i) * max_rows + s) * kDim);
    float* dsc = scales_out + (size_t(i) * max_rows + s) * kScales;
    if (ref.row >= 0) {
      const uint4* src = reinterpret_cast<const uint4*>(ref.kv);
      for (int j = 0; j < kDim / 16; ++j) dst[j] = src[j];
      for (int j = 0; j < kScales; ++j) dsc[j] = ref.sc[j];
      row_ids_out[size_t(i) * max_rows + s] = (ref.source << 30) | ref.row;
    } else {
      for (int j = 0; j < kDim / 16; ++j) dst[j] = make_uint4(0, 0, 0, 0);
      for (int j = 0; j < kScales; ++j) dsc[j] = 0.f;
      row_ids_out[size_t(i) * max_rows + s] = -1;
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

cudaError_t launch_plan(const qsfm_params& p, int num_tokens, int num_ctas, int split,
                        int32_t* metadata, int* fault, cudaStream_t s) {
  (void)fault;
  plan_kernel<<<1, kPlanThreads, 0, s>>>(p, num_tokens, num_ctas, split, metadata);
  return cudaGetLastError();
}

cudaError_t launch_combine(const qsfm_params& p, int num_tokens, int num_ctas,
                           const Workspace& ws, int* fault, cudaStream_t s) {
  combine_kernel<<<num_ctas, 256, 0, s>>>(p, num_tokens, ws, fault);
  return cudaGetLastError();
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
