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
// Both accumulators live in tensor memory: S^T in 64 columns, O^T in 256
// columns. One dequantised bf16 tile in shared memory (128 rows x 512, 128-B
// swizzle) is the K-major A operand of the first product and the MN-major A
// operand of the second.
//
// Per tile: gather 128 paged fp8 rows + their per-64 scales -> dequantise to
// bf16 in the swizzled layout -> tcgen05 QK^T -> masked online softmax in
// registers (thread = KV row; per-head max / sum over rows by warp
// butterflies and a 4-warp exchange) -> P^T to shared memory -> tcgen05 PV.
// The running max is only moved when a tile's max exceeds it by more than
// 2^8 (exact: the rescale is applied to O and l whenever it is moved).
#include <cuda_runtime.h>

#include "qsfm_device.cuh"
#include "qsfm_internal.h"

namespace qsfm {
namespace {

constexpr int kThreads = 128;
// shared memory map (byte offsets from a 1024-aligned base)
constexpr uint32_t kSK = 0;                        // K~: 8 d-blocks x 128 rows x 128 B
constexpr uint32_t kSQ = kSK + 8 * 128 * 128;      // Q: 8 d-blocks x 64 heads x 128 B
constexpr uint32_t kSP = kSQ + 8 * 64 * 128;       // P^T: 128 rows x 64 heads (bf16)
constexpr uint32_t kSRed = kSP + 128 * 128;        // red_max[4][64], red_sum[4][64]
constexpr uint32_t kSStat = kSRed + 2 * 4 * 64 * 4;  // m_used, l_run, alpha, inv [64] each
constexpr uint32_t kSValid = kSStat + 4 * 64 * 4;  // row valid flags [128]
constexpr uint32_t kSBar = kSValid + 128 * 4;      // 2 mbarriers, tmem base, flags
constexpr uint32_t kSmemBytes = kSBar + 64;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = 256;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kIdescQK = make_idesc_bf16(128, 64, /*a_mn=*/0, /*b_mn=*/0);
constexpr uint32_t kIdescPV = make_idesc_bf16(128, 64, /*a_mn=*/1, /*b_mn=*/1);
constexpr uint32_t kWaitIters = 1u << 26;

// Reduce 64 per-thread values over the 32 lanes of a warp. Afterwards lane l
// holds the result for heads 2l and 2l+1 in r0 / r1.
template <bool kMax>
__device__ __forceinline__ void warp_reduce64(const float (&v)[64], float& r0, float& r1) {
  const int lane = threadIdx.x & 31;
  float a[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const bool up = lane & 16;
    const float keep = up ? v[32 + i] : v[i];
    const float send = up ? v[i] : v[32 + i];
    const float got = __shfl_xor_sync(0xffffffffu, send, 16);
    a[i] = kMax ? fmaxf(keep, got) : keep + got;
  }
  float b[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const bool up = lane & 8;
    const float keep = up ? a[16 + i] : a[i];
    const float send = up ? a[i] : a[16 + i];
    const float got = __shfl_xor_sync(0xffffffffu, send, 8);
    b[i] = kMax ? fmaxf(keep, got) : keep + got;
  }
  float c[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool up = lane & 4;
    const float keep = up ? b[8 + i] : b[i];
    const float send = up ? b[i] : b[8 + i];
    const float got = __shfl_xor_sync(0xffffffffu, send, 4);
    c[i] = kMax ? fmaxf(keep, got) : keep + got;
  }
  float d[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool up = lane & 2;
    const float keep = up ? c[4 + i] : c[i];
    const float send = up ? c[i] : c[4 + i];
    const float got = __shfl_xor_sync(0xffffffffu, send, 2);
    d[i] = kMax ? fmaxf(keep, got) : keep + got;
  }
  float e[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool up = lane & 1;
    const float keep = up ? d[2 + i] : d[i];
    const float send = up ? d[i] : d[2 + i];
    const float got = __shfl_xor_sync(0xffffffffu, send, 1);
    e[i] = kMax ? fmaxf(keep, got) : keep + got;
  }
  r0 = e[0];
  r1 = e[1];
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(kThreads, 1)
    attention_kernel(const qsfm_params p, const int T, const Workspace ws, int* fault) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_addr);
  float* red_max = reinterpret_cast<float*>(smem + kSRed);
  float* red_sum = red_max + 4 * 64;
  float* m_used = reinterpret_cast<float*>(smem + kSStat);
  float* l_run = m_used + 64;
  float* alpha = l_run + 64;
  float* inv = alpha + 64;
  int* row_valid = reinterpret_cast<int*>(smem + kSValid);
  uint64_t* bar_s = reinterpret_cast<uint64_t*>(smem + kSBar);
  uint64_t* bar_o = bar_s + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSBar + 16);
  volatile int* flags = reinterpret_cast<volatile int*>(smem + kSBar + 32);  // [0] rescale [1] abort

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
  const int t0 = meta[kMetaHeader + 2 * c], k0 = meta[kMetaHeader + 2 * c + 1];
  const int t1 = meta[kMetaHeader + 2 * c + 2], k1 = meta[kMetaHeader + 2 * c + 3];
  if (t0 < 0 || t1 > T || t0 > t1 || k0 < 0 || k1 < 0 || (t1 == T && k1 != 0)) {
    if (tid == 0) atomicOr(fault, QSFM_FAULT_METADATA);
    return;
  }
  if (t0 == t1 && k0 == k1) return;

  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    fence_mbar_init();
    flags[0] = 0;
    flags[1] = 0;
  }
  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = uint32_t(warp * 32) << 16;
  const float qk_scale = p.softmax_scale * kLog2e;
  uint32_t ph_s = 0, ph_o = 0;
  bool aborted = false;

  for (int t = t0; t <= t1 && t < T && !aborted; ++t) {
    if (t == t1 && k1 == 0) break;
    const TokenGeom g = token_geom(p, t);
    const int klo = (t == t0) ? min(k0, g.n_tiles) : 0;
    const int khi = (t == t1) ? min(k1, g.n_tiles) : g.n_tiles;
    const bool whole = (klo == 0 && khi == g.n_tiles);
    const int slot = (t == t0) ? 2 * c : 2 * c + 1;
    if (!whole && slot >= ws.slots) {  // plan splits a token but no workspace was given
      if (tid == 0) atomicOr(fault, QSFM_FAULT_METADATA);
      break;
    }

    if (tid < 64) {
      m_used[tid] = -INFINITY;
      l_run[tid] = 0.f;
    }
    // Q of the token -> swizzled K-major [8 d-blocks][64 heads][128 B]
    if (klo < khi) {
      const uint8_t* qg = static_cast<const uint8_t*>(p.q) + size_t(t) * kHeads * kDim * 2;
#pragma unroll 4
      for (int i = tid; i < kHeads * kDim / 8; i += kThreads) {
        const int h = i >> 6, c16 = i & 63;
        const uint4 v = ldg_nc_v4(qg + size_t(i) * 16);
        sts_v4(sbase + kSQ + (c16 >> 3) * 8192 + h * 128 + (((c16 & 7) ^ (h & 7)) << 4), v);
      }
    }

    bool first = true;
    for (int k = klo; k < khi; ++k) {
      // ---- gather + dequantise 128 rows into the swizzled tile
#pragma unroll 1
      for (int gi = 0; gi < 4; ++gi) {
        const int r = warp * 32 + gi * 8 + (lane & 7);
        const RowRef ref = resolve_slot(p, g, t, k, r, fault);
        const bool valid = ref.row >= 0;
        if ((lane >> 3) == 0) row_valid[r] = valid ? 1 : 0;
        const uint32_t sw = uint32_t(r & 7);
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
          const int u = pp * 4 + (lane >> 3);
          const uint32_t dst = sbase + kSK + u * 16384 + r * 128;
          if (valid) {
            const uint8_t* src = ref.kv + u * 64;
            const float sc = __ldg(ref.sc + u);
            uint4 in[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) in[m] = ldg_nc_v4(src + 16 * m);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              uint4 lo, hi;
              dequant16(in[m], sc, lo, hi);
              sts_v4(dst + (((2 * m) ^ sw) << 4), lo);
              sts_v4(dst + (((2 * m + 1) ^ sw) << 4), hi);
            }
          } else {
            const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) sts_v4(dst + ((ch ^ sw) << 4), z);
          }
        }
      }
      fence_proxy_async_smem();
      __syncthreads();

      // ---- S^T = K~ Q^T
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t a = make_sdesc_sw128(sbase + kSK + kb * 16384 + kk * 32, 16, 1024);
            const uint64_t b = make_sdesc_sw128(sbase + kSQ + kb * 8192 + kk * 32, 16, 1024);
            mma_bf16(tmem + kTmemS, a, b, kIdescQK, (kb | kk) != 0);
          }
        }
        mma_commit(bar_s);
        if (!mbar_wait(bar_s, ph_s, kWaitIters)) {
          flags[1] = 1;
          atomicOr(fault, QSFM_FAULT_TIMEOUT);
        }
      }
      ph_s ^= 1;
      __syncthreads();
      if (flags[1]) { aborted = true; break; }
      tc_fence_after();

      // ---- masked online softmax (thread = KV row of the tile)
      float x[64];
#pragma unroll
      for (int j = 0; j < 4; ++j) tmem_ld16(tmem + kTmemS + lane_base + j * 16, x + j * 16);
      tmem_ld_wait();
      const bool rv = row_valid[tid] != 0;
#pragma unroll
      for (int h = 0; h < 64; ++h) x[h] = rv ? x[h] * qk_scale : -INFINITY;
      float r0, r1;
      warp_reduce64<true>(x, r0, r1);
      red_max[warp * 64 + 2 * lane] = r0;
      red_max[warp * 64 + 2 * lane + 1] = r1;
      __syncthreads();
      if (tid < 64) {
        const float mt = fmaxf(fmaxf(red_max[tid], red_max[64 + tid]),
                               fmaxf(red_max[128 + tid], red_max[192 + tid]));
        const float mu = m_used[tid];
        float a = 1.f;
        if (mt > -INFINITY && (mu == -INFINITY || mt > mu + kRescaleLog2)) {
          a = (mu == -INFINITY) ? 0.f : exp2f(mu - mt);
          m_used[tid] = mt;
          if (!first) flags[0] = 1;
        }
        alpha[tid] = a;
      }
      __syncthreads();
      float pr[64];
#pragma unroll
      for (int h = 0; h < 64; ++h) {
        const float mu = m_used[h];
        pr[h] = exp2f(x[h] - (mu == -INFINITY ? 0.f : mu));
      }
      warp_reduce64<false>(pr, r0, r1);
      red_sum[warp * 64 + 2 * lane] = r0;
      red_sum[warp * 64 + 2 * lane + 1] = r1;
      {
        const uint32_t prow = sbase + kSP + tid * 128;
        const uint32_t sw = uint32_t(tid & 7);
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          uint4 v;
          v.x = pack_bf16(pr[8 * cc + 0], pr[8 * cc + 1]);
          v.y = pack_bf16(pr[8 * cc + 2], pr[8 * cc + 3]);
          v.z = pack_bf16(pr[8 * cc + 4], pr[8 * cc + 5]);
          v.w = pack_bf16(pr[8 * cc + 6], pr[8 * cc + 7]);
          sts_v4(prow + ((uint32_t(cc) ^ sw) << 4), v);
        }
      }
      __syncthreads();
      if (tid < 64) {
        l_run[tid] = l_run[tid] * alpha[tid] + (red_sum[tid] + red_sum[64 + tid]) +
                     (red_sum[128 + tid] + red_sum[192 + tid]);
      }
      if (flags[0]) {  // move O^T to the new running max (previous PV has completed)
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float o[16];
            const uint32_t addr = tmem + kTmemO + cc * 64 + j * 16 + lane_base;
            tmem_ld16(addr, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] *= alpha[j * 16 + i];
            tmem_st16(addr, o);
          }
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) flags[0] = 0;

      // ---- O^T += V~^T P^T
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t a = make_sdesc_sw128(sbase + kSK + cc * 32768 + ks * 2048, 16384, 1024);
            const uint64_t b = make_sdesc_sw128(sbase + kSP + ks * 2048, 16, 1024);
            mma_bf16(tmem + kTmemO + cc * 64, a, b, kIdescPV, (first && ks == 0) ? 0u : 1u);
          }
        }
        mma_commit(bar_o);
        if (!mbar_wait(bar_o, ph_o, kWaitIters)) {
          flags[1] = 1;
          atomicOr(fault, QSFM_FAULT_TIMEOUT);
        }
      }
      ph_o ^= 1;
      __syncthreads();
      if (flags[1]) { aborted = true; break; }
      tc_fence_after();
      first = false;
    }
    if (aborted) break;

    // ---- epilogue: normalise, add the sink (whole tokens), write out
    const bool any = !first;  // at least one tile went through the MMAs
    if (tid < 64) {
      const float l = l_run[tid], mu = m_used[tid];
      const float lse2 = l > 0.f ? mu + log2f(l) : -INFINITY;
      if (whole) {
        float den = l;
        if (p.sinks != nullptr && l > 0.f) den += exp2f(__ldg(p.sinks + tid) * kLog2e - mu);
        inv[tid] = l > 0.f ? 1.f / den : 0.f;
        if (p.return_lse) p.softmax_lse[size_t(t) * 64 + tid] = lse2 * kLn2;
      } else {
        inv[tid] = l > 0.f ? 1.f / l : 0.f;
        ws.lse[size_t(slot) * 64 + tid] = lse2 * kLn2;
      }
    }
    __syncthreads();
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      float o[64];
      if (any) {
#pragma unroll
        for (int j = 0; j < 4; ++j) tmem_ld16(tmem + kTmemO + cc * 64 + j * 16 + lane_base, o + j * 16);
        tmem_ld_wait();
      }
      const int d = cc * 128 + warp * 32 + lane;
      if (whole) {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.attn_out) + size_t(t) * 64 * kDim + d;
#pragma unroll
        for (int h = 0; h < 64; ++h) out[size_t(h) * kDim] = __float2bfloat16_rn(any ? o[h] * inv[h] : 0.f);
      } else {
        float* out = ws.out + size_t(slot) * 64 * kDim + d;
#pragma unroll
        for (int h = 0; h < 64; ++h) out[size_t(h) * kDim] = any ? o[h] * inv[h] : 0.f;
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_attention(const qsfm_params& p, int num_tokens, int num_ctas,
                             const Workspace& ws, int* fault, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(attention_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
  if (e != cudaSuccess) return e;
  attention_kernel<<<num_ctas, kThreads, kSmemAlloc, s>>>(p, num_tokens, ws, fault);
  return cudaGetLastError();
}

}  // namespace qsfm
