// C-ABI entry points: argument validation on the host, then kernel launches
// on the caller's stream. Nothing here reads device memory back, so every
// call can be captured in a CUDA graph (QuantSparseFlashMla, constraints:
// aclgraph mode is supported).
//
// Validation follows QuantSparseFlashMla's constraints section: N2 = 1 and
// D = 512; cmp_ratio in [1, 128] and 1 when only ori_kv is passed; ori mask
// mode 0/3/4 and cmp mask mode 0/3; windows -1 or >= 0, and >= 0 only with
// ori mask mode 4; cu_seqlens_q required for TND; seqused_ori_kv and the
// block table required for paged KV; metadata required.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "qsfm.h"
#include "qsfm_internal.h"

namespace {

// Device fault word (QSFM_FAULT_* bits), one per device that loads the
// library. Kernels get its address as an argument.
__device__ int g_fault_word;

// The address is looked up once per device, under a lock: two host threads
// making their first call on a device at the same time both see it set.
std::mutex g_fault_lock;

int* fault_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  static int* ptrs[64] = {nullptr};
  std::lock_guard<std::mutex> guard(g_fault_lock);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fault_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

int num_tokens(const qsfm_params& p) {
  return p.layout_q == QSFM_LAYOUT_BSND ? p.batch * p.max_s1 : p.total_t;
}

// Work units the kernels plan over: one per 64-head group of each token
// (N1 = 64: the tokens; N1 = 128: two per token).
int num_units(const qsfm_params& p) { return num_tokens(p) * (p.n1 / QSFM_NUM_HEADS); }

// CTAs the work is planned over: p.num_ctas, or the SM count when 0. With at
// least as many tokens as CTAs the plan cuts at token starts, so some CTAs
// get ceil(T / n) tokens; the fewest CTAs that keep that maximum take their
// place (256 tokens on 152 SMs: 128 CTAs of 2 tokens instead of 104 CTAs of
// 2 and 48 of 1). The longest CTA does as much work as before while fewer
// CTAs compete for memory and L2.
qsfm_status resolve_ctas(const qsfm_params& p, int* out) {
  int n = p.num_ctas;
  if (n <= 0) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QSFM_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return QSFM_ERR_CUDA;
    n = sms < QSFM_MAX_CTAS ? sms : QSFM_MAX_CTAS;
  }
  const long long T = num_units(p);
  if (T >= n) {
    const long long per = (T + n - 1) / n;
    n = int((T + per - 1) / per);
  }
  *out = n;
  return QSFM_OK;
}

// Limits of the kernels' 32-bit index arithmetic (work units, head rows,
// index offsets within a row, physical KV rows). Every batch that fits in
// device memory is far below them; larger shapes are refused, not wrapped.
constexpr long long kMaxUnits = 1ll << 24;     // units x 64 head rows < 2^31
constexpr int kMaxK2 = 1 << 16;                // index entries per token
constexpr long long kMaxPoolRows = (1ll << 31) - 1;

// True for a null pointer or one aligned to `bytes`.
bool aligned(const void* ptr, uintptr_t bytes) {
  return (reinterpret_cast<uintptr_t>(ptr) & (bytes - 1)) == 0;
}

// Shape / attribute / pointer checks shared by every entry point.
qsfm_status validate(const qsfm_params* pp, bool need_outputs) {
  if (pp == nullptr) return QSFM_ERR_INVALID_ARG;
  const qsfm_params& p = *pp;
  if (p.n1 <= 0 || p.d <= 0) return QSFM_ERR_INVALID_ARG;
  if (p.d != QSFM_HEAD_DIM) return QSFM_ERR_INVALID_ARG;  // "D only supports 512"
  if (p.n1 != QSFM_NUM_HEADS && p.n1 != 2 * QSFM_NUM_HEADS) return QSFM_ERR_UNSUPPORTED;
  if (p.batch < 0) return QSFM_ERR_INVALID_ARG;
  if (p.layout_q != QSFM_LAYOUT_BSND && p.layout_q != QSFM_LAYOUT_TND) return QSFM_ERR_INVALID_ARG;
  if (p.layout_q == QSFM_LAYOUT_BSND && p.max_s1 < 0) return QSFM_ERR_INVALID_ARG;
  if (p.layout_q == QSFM_LAYOUT_TND) {
    if (p.total_t < 0) return QSFM_ERR_INVALID_ARG;
    if (p.cu_seqlens_q == nullptr && p.batch > 0) return QSFM_ERR_INVALID_ARG;
  }
  if (p.num_ctas < 0 || p.num_ctas > QSFM_MAX_CTAS) return QSFM_ERR_INVALID_ARG;
  const long long tokens = p.layout_q == QSFM_LAYOUT_BSND ? (long long)p.batch * p.max_s1 : p.total_t;
  if (tokens * (p.n1 / QSFM_NUM_HEADS) > kMaxUnits) return QSFM_ERR_UNSUPPORTED;
  if (p.k2 < 0) return QSFM_ERR_INVALID_ARG;
  if (p.k2 > kMaxK2) return QSFM_ERR_UNSUPPORTED;
  if (p.kv_layout != QSFM_KV_FP8_FP32_SCALES && p.kv_layout != QSFM_KV_PACKED640 &&
      p.kv_layout != QSFM_KV_BF16)
    return QSFM_ERR_INVALID_ARG;
  const bool no_scales = p.kv_layout != QSFM_KV_FP8_FP32_SCALES;
  // packed rows carry their scales and bf16 rows need none: a separate scale
  // tensor with them is a mistake
  if (no_scales && (p.ori_scale != nullptr || p.cmp_scale != nullptr)) return QSFM_ERR_INVALID_ARG;
  if (p.ori_kv == nullptr || (!no_scales && p.ori_scale == nullptr)) return QSFM_ERR_INVALID_ARG;
  if (p.cmp_ratio < 1 || p.cmp_ratio > 128) return QSFM_ERR_INVALID_ARG;
  if (p.cmp_kv == nullptr) {
    if (p.cmp_ratio != 1) return QSFM_ERR_INVALID_ARG;  // SWA keeps the default 1
    if (p.cmp_sparse_indices != nullptr) return QSFM_ERR_INVALID_ARG;  // CSA needs cmp_kv
  } else if (!no_scales && p.cmp_scale == nullptr) {
    return QSFM_ERR_INVALID_ARG;
  }
  // KV storage (QuantSparseFlashMla constraints on layout_kv): BSND / TND KV
  // only with the same q layout; block tables and seqused_ori_kv only where
  // the layout uses them
  if (p.layout_kv == QSFM_LAYOUT_KV_PA_BBND) {
    if (p.cu_seqlens_ori_kv != nullptr || p.cu_seqlens_cmp_kv != nullptr) return QSFM_ERR_INVALID_ARG;
    if (p.ori_block_size < 1 || p.ori_block_size > 1024) return QSFM_ERR_INVALID_ARG;
    if (p.ori_block_size != QSFM_BLOCK_SIZE) return QSFM_ERR_UNSUPPORTED;
    if (p.ori_block_table == nullptr || p.seqused_ori_kv == nullptr) return QSFM_ERR_INVALID_ARG;
    if (p.ori_max_blocks < 1 || p.ori_num_blocks < 1) return QSFM_ERR_INVALID_ARG;
    if ((long long)p.ori_num_blocks * p.ori_block_size > kMaxPoolRows) return QSFM_ERR_UNSUPPORTED;
    if (p.cmp_kv != nullptr) {
      if (p.cmp_block_size < 1 || p.cmp_block_size > 1024) return QSFM_ERR_INVALID_ARG;
      if (p.cmp_block_size != QSFM_BLOCK_SIZE) return QSFM_ERR_UNSUPPORTED;
      if (p.cmp_block_table == nullptr) return QSFM_ERR_INVALID_ARG;
      if (p.cmp_max_blocks < 1 || p.cmp_num_blocks < 1) return QSFM_ERR_INVALID_ARG;
      if ((long long)p.cmp_num_blocks * p.cmp_block_size > kMaxPoolRows) return QSFM_ERR_UNSUPPORTED;
    }
  } else if (p.layout_kv == QSFM_LAYOUT_KV_BSND || p.layout_kv == QSFM_LAYOUT_KV_TND) {
    const bool tnd = p.layout_kv == QSFM_LAYOUT_KV_TND;
    if (p.layout_q != (tnd ? QSFM_LAYOUT_TND : QSFM_LAYOUT_BSND)) return QSFM_ERR_INVALID_ARG;
    if (p.ori_block_table != nullptr || p.cmp_block_table != nullptr) return QSFM_ERR_INVALID_ARG;
    if (p.ori_kv_len < 1 || (p.cmp_kv != nullptr && p.cmp_kv_len < 1)) return QSFM_ERR_INVALID_ARG;
    if (tnd) {
      if (p.seqused_ori_kv != nullptr || (p.cu_seqlens_ori_kv == nullptr && p.batch > 0))
        return QSFM_ERR_INVALID_ARG;
      if (p.cmp_kv != nullptr && p.cu_seqlens_cmp_kv == nullptr && p.batch > 0) return QSFM_ERR_INVALID_ARG;
      if (p.cmp_kv == nullptr && p.cu_seqlens_cmp_kv != nullptr) return QSFM_ERR_INVALID_ARG;
    } else {
      if (p.cu_seqlens_ori_kv != nullptr || p.cu_seqlens_cmp_kv != nullptr) return QSFM_ERR_INVALID_ARG;
      // rows b * S + j of the whole tensor stay below 2^31
      if ((long long)p.batch * p.ori_kv_len > kMaxPoolRows) return QSFM_ERR_UNSUPPORTED;
      if (p.cmp_kv != nullptr && (long long)p.batch * p.cmp_kv_len > kMaxPoolRows) return QSFM_ERR_UNSUPPORTED;
    }
  } else {
    return QSFM_ERR_INVALID_ARG;
  }
  if (p.cmp_sparse_indices != nullptr && p.k2 < 1) return QSFM_ERR_INVALID_ARG;
  // discrete ori picks (QuantSparseFlashMla parameter table rows
  // ori_sparse_indices and ori_topk_length)
  if (p.ori_sparse_indices != nullptr) {
    if (p.k1 < 1) return QSFM_ERR_INVALID_ARG;
    if (p.k1 > kMaxK2) return QSFM_ERR_UNSUPPORTED;
  } else if (p.k1 != 0 || p.ori_topk_length != nullptr) {
    return QSFM_ERR_INVALID_ARG;
  }
  if (p.ori_mask_mode != 0 && p.ori_mask_mode != 3 && p.ori_mask_mode != 4)
    return QSFM_ERR_INVALID_ARG;
  if (p.cmp_mask_mode != 0 && p.cmp_mask_mode != 3) return QSFM_ERR_INVALID_ARG;
  if (p.ori_win_left < -1 || p.ori_win_right < -1) return QSFM_ERR_INVALID_ARG;
  if (p.ori_mask_mode != 4 && (p.ori_win_left >= 0 || p.ori_win_right >= 0))
    return QSFM_ERR_INVALID_ARG;
  if (!std::isfinite(p.softmax_scale)) return QSFM_ERR_INVALID_ARG;
  if (need_outputs && num_tokens(p) > 0) {
    if (p.q == nullptr || p.attn_out == nullptr) return QSFM_ERR_INVALID_ARG;
    if (p.return_lse && p.softmax_lse == nullptr) return QSFM_ERR_INVALID_ARG;
  }
  // Alignment the kernels rely on: 16-byte vector, tensor-map and bulk-copy
  // accesses to q, the KV pools and attn_out; 4-byte element accesses to the
  // rest.
  if (!aligned(p.q, 16) || !aligned(p.ori_kv, 16) || !aligned(p.cmp_kv, 16) ||
      !aligned(p.attn_out, 16))
    return QSFM_ERR_INVALID_ARG;
  const void* words[] = {p.ori_scale, p.cmp_scale, p.cmp_sparse_indices, p.ori_block_table,
                         p.cmp_block_table, p.cu_seqlens_q, p.seqused_q, p.seqused_ori_kv,
                         p.seqused_cmp_kv, p.cmp_residual_kv, p.cmp_topk_length, p.sinks,
                         p.metadata, p.softmax_lse, p.cu_seqlens_ori_kv, p.cu_seqlens_cmp_kv,
                         p.ori_sparse_indices, p.ori_topk_length};
  for (const void* w : words)
    if (!aligned(w, 4)) return QSFM_ERR_INVALID_ARG;
  return QSFM_OK;
}

// Whether the plan may cut inside a token: only when there are fewer query
// tokens than CTAs (decode); longer batches are cut at token starts.
int split_mode(int tokens, int ctas) { return tokens < ctas ? 1 : 0; }

// The last CUDA runtime error an entry point returned QSFM_ERR_CUDA for, on
// this host thread (read by qsfm_last_cuda_error).
thread_local int g_last_cuda_error = 0;

qsfm_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return QSFM_OK;
  g_last_cuda_error = int(e);
  return QSFM_ERR_CUDA;
}

// A named NVTX range around each launch, so that a profiler timeline shows
// which entry point a kernel belongs to. With no tool attached a range costs
// one indirect call; nothing is recorded.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

qsfm_status prepare_forward(const qsfm_params* p, void* workspace, size_t ws_bytes, int* ctas,
                            qsfm::Workspace* ws, int** fault) {
  qsfm_status st = validate(p, true);
  if (st != QSFM_OK) return st;
  if (p->metadata == nullptr) return QSFM_ERR_INVALID_ARG;
  st = resolve_ctas(*p, ctas);
  if (st != QSFM_OK) return st;
  const int T = num_units(*p);
  if (split_mode(T, *ctas)) {
    if (workspace == nullptr || ws_bytes < qsfm::workspace_bytes(*ctas)) return QSFM_ERR_WORKSPACE;
    *ws = qsfm::workspace_view(workspace, *ctas);
  } else {
    *ws = qsfm::Workspace{nullptr, nullptr, 0};
  }
  *fault = fault_ptr();
  if (*fault == nullptr) return QSFM_ERR_CUDA;
  return QSFM_OK;
}

}  // namespace

namespace {

constexpr long long kMaxIndexerTokens = 1ll << 20;

// Checks shared by the indexer's size query and launch; *T gets the query
// rows.
qsfm_status check_indexer(const qsfm_indexer_params* pp, long long* T) {
  if (pp == nullptr || T == nullptr) return QSFM_ERR_INVALID_ARG;
  const qsfm_indexer_params& p = *pp;
  if (p.batch < 0 || p.heads < 1 || p.dim < 1 || p.topk < 1) return QSFM_ERR_INVALID_ARG;
  if (p.heads > 64 || p.topk > 8192) return QSFM_ERR_INVALID_ARG;
  if (p.dim != 128) return QSFM_ERR_UNSUPPORTED;
  if (p.block_size < 1 || p.block_size > 1024) return QSFM_ERR_INVALID_ARG;
  if (p.block_size != QSFM_BLOCK_SIZE) return QSFM_ERR_UNSUPPORTED;
  if (p.mask_mode != 0 && p.mask_mode != 3) return QSFM_ERR_INVALID_ARG;
  if (p.cmp_ratio < 1 || p.cmp_ratio > 128) return QSFM_ERR_INVALID_ARG;
  if (p.layout_q == QSFM_LAYOUT_BSND) {
    if (p.max_s1 < 0 || p.cu_seqlens_q != nullptr) return QSFM_ERR_INVALID_ARG;
  } else if (p.layout_q == QSFM_LAYOUT_TND) {
    if (p.total_t < 0 || (p.cu_seqlens_q == nullptr && p.batch > 0)) return QSFM_ERR_INVALID_ARG;
  } else {
    return QSFM_ERR_INVALID_ARG;
  }
  // key layouts (parameter table: layout_k, seqused_k, cu_seqlens_k,
  // block_table): the paged layout takes the table and seqused_k, BSND
  // slabs an optional seqused_k, TND rows cu_seqlens_k and no seqused_k
  if (p.layout_k == QSFM_LAYOUT_KV_PA_BBND) {
    if (p.max_blocks < 1 || p.num_blocks < 1 || p.cu_seqlens_k != nullptr) return QSFM_ERR_INVALID_ARG;
  } else if (p.layout_k == QSFM_LAYOUT_KV_BSND) {
    if (p.max_sk < 0 || p.block_table != nullptr || p.cu_seqlens_k != nullptr) return QSFM_ERR_INVALID_ARG;
    if ((long long)p.batch * p.max_sk > kMaxPoolRows) return QSFM_ERR_UNSUPPORTED;
  } else if (p.layout_k == QSFM_LAYOUT_KV_TND) {
    if (p.total_k < 0 || p.block_table != nullptr || p.seqused_k != nullptr ||
        (p.cu_seqlens_k == nullptr && p.batch > 0))
      return QSFM_ERR_INVALID_ARG;
  } else {
    return QSFM_ERR_INVALID_ARG;
  }
  *T = p.layout_q == QSFM_LAYOUT_BSND ? (long long)p.batch * p.max_s1 : p.total_t;
  if (*T > kMaxIndexerTokens) return QSFM_ERR_UNSUPPORTED;
  return QSFM_OK;
}

}  // namespace

extern "C" {

void qsfm_params_init(qsfm_params* p) {
  if (p == nullptr) return;
  std::memset(p, 0, sizeof(*p));
  p->n1 = QSFM_NUM_HEADS;
  p->d = QSFM_HEAD_DIM;
  p->ori_block_size = QSFM_BLOCK_SIZE;
  p->cmp_block_size = QSFM_BLOCK_SIZE;
  p->softmax_scale = 1.0f / std::sqrt(float(QSFM_HEAD_DIM));
  p->cmp_ratio = 1;
  p->ori_mask_mode = 4;
  p->cmp_mask_mode = 3;
  p->ori_win_left = 127;
  p->ori_win_right = 0;
  p->layout_q = QSFM_LAYOUT_BSND;
}

qsfm_status qsfm_metadata(const qsfm_params* p, int32_t* metadata_out, void* stream) {
  qsfm_status st = validate(p, false);
  if (st != QSFM_OK) return st;
  if (metadata_out == nullptr || !aligned(metadata_out, 4)) return QSFM_ERR_INVALID_ARG;
  int ctas = 0;
  st = resolve_ctas(*p, &ctas);
  if (st != QSFM_OK) return st;
  int* fault = fault_ptr();
  if (fault == nullptr) return QSFM_ERR_CUDA;
  const int T = num_units(*p);
  const NvtxRange range("qsfm_metadata");
  return cuda_status(qsfm::launch_plan(*p, T, ctas, split_mode(T, ctas), metadata_out, fault,
                                       static_cast<cudaStream_t>(stream)));
}

qsfm_status qsfm_forward_workspace_size(const qsfm_params* p, size_t* bytes) {
  qsfm_status st = validate(p, false);
  if (st != QSFM_OK) return st;
  if (bytes == nullptr) return QSFM_ERR_INVALID_ARG;
  int ctas = 0;
  st = resolve_ctas(*p, &ctas);
  if (st != QSFM_OK) return st;
  *bytes = split_mode(num_units(*p), ctas) ? qsfm::workspace_bytes(ctas) : 0;
  return QSFM_OK;
}

qsfm_status qsfm_attention(const qsfm_params* p, void* workspace, size_t workspace_bytes,
                           void* stream) {
  int ctas = 0;
  qsfm::Workspace ws{};
  int* fault = nullptr;
  qsfm_status st = prepare_forward(p, workspace, workspace_bytes, &ctas, &ws, &fault);
  if (st != QSFM_OK) return st;
  const int T = num_units(*p);
  if (T == 0) return QSFM_OK;
  const NvtxRange range("qsfm_attention");
  return cuda_status(
      qsfm::launch_attention(*p, T, ctas, ws, fault, static_cast<cudaStream_t>(stream)));
}

qsfm_status qsfm_combine(const qsfm_params* p, void* workspace, size_t workspace_bytes,
                         void* stream) {
  int ctas = 0;
  qsfm::Workspace ws{};
  int* fault = nullptr;
  qsfm_status st = prepare_forward(p, workspace, workspace_bytes, &ctas, &ws, &fault);
  if (st != QSFM_OK) return st;
  const int T = num_units(*p);
  if (T == 0 || !split_mode(T, ctas)) return QSFM_OK;  // no token can be split
  const NvtxRange range("qsfm_combine");
  return cuda_status(
      qsfm::launch_combine(*p, T, ctas, ws, fault, static_cast<cudaStream_t>(stream)));
}

qsfm_status qsfm_forward(const qsfm_params* p, void* workspace, size_t workspace_bytes,
                         void* stream) {
  qsfm_status st = qsfm_attention(p, workspace, workspace_bytes, stream);
  if (st != QSFM_OK) return st;
  return qsfm_combine(p, workspace, workspace_bytes, stream);
}

qsfm_status qsfm_debug_gather(const qsfm_params* p, const int32_t* tokens, int32_t n,
                              int32_t max_rows, uint8_t* rows_out, float* scales_out,
                              int32_t* row_ids_out, int32_t* counts_out, void* stream) {
  qsfm_status st = validate(p, false);
  if (st != QSFM_OK) return st;
  // row bytes are exported in the pool's own row format; separate scales
  // exist for fp8 rows only. With rows_out = scales_out = NULL only the row
  // ids and counts are written.
  const bool fp8 = p->kv_layout == QSFM_KV_FP8_FP32_SCALES;
  if (!fp8 && scales_out != nullptr) return QSFM_ERR_INVALID_ARG;
  if (fp8 && (rows_out == nullptr) != (scales_out == nullptr)) return QSFM_ERR_INVALID_ARG;
  if (n < 0 || max_rows < 0) return QSFM_ERR_INVALID_ARG;
  if (n == 0) return QSFM_OK;
  if (tokens == nullptr || counts_out == nullptr) return QSFM_ERR_INVALID_ARG;
  if (max_rows > 0 && row_ids_out == nullptr) return QSFM_ERR_INVALID_ARG;
  if (!aligned(rows_out, 16)) return QSFM_ERR_INVALID_ARG;
  int* fault = fault_ptr();
  if (fault == nullptr) return QSFM_ERR_CUDA;
  return cuda_status(qsfm::launch_debug_gather(*p, tokens, n, max_rows, rows_out, scales_out,
                                               row_ids_out, counts_out, fault,
                                               static_cast<cudaStream_t>(stream)));
}

qsfm_status qsfm_debug_bounded_wait(uint64_t timeout_ns, uint64_t* elapsed_ns_out, void* stream) {
  if (elapsed_ns_out == nullptr || !aligned(elapsed_ns_out, 8)) return QSFM_ERR_INVALID_ARG;
  if (timeout_ns == 0 || timeout_ns > 1000000000ull) return QSFM_ERR_INVALID_ARG;
  int* fault = fault_ptr();
  if (fault == nullptr) return QSFM_ERR_CUDA;
  return cuda_status(qsfm::launch_bounded_wait(
      timeout_ns, reinterpret_cast<unsigned long long*>(elapsed_ns_out), fault,
      static_cast<cudaStream_t>(stream)));
}

void qsfm_indexer_params_init(qsfm_indexer_params* p) {
  if (p == nullptr) return;
  std::memset(p, 0, sizeof(*p));
  p->heads = 64;
  p->dim = 128;
  p->topk = 2048;  // QuantLightningIndexerV2 parameter table: topk default
  p->block_size = QSFM_BLOCK_SIZE;
  p->cmp_ratio = 1;
  p->layout_q = QSFM_LAYOUT_BSND;
}

// QuantLightningIndexerV2 constraints: query N in [1, 64], key N = 1, topk
// in [1, 8192]; quant mode 1 (e4m3 query / key, fp32 scales and weights);
// cu_seqlens_q required for TND and not allowed for BSND.
qsfm_status qsfm_lightning_indexer_workspace_size(const qsfm_indexer_params* p, size_t* bytes) {
  if (bytes == nullptr) return QSFM_ERR_INVALID_ARG;
  long long T = 0;
  const qsfm_status st = check_indexer(p, &T);
  if (st != QSFM_OK) return st;
  *bytes = qsfm::indexer_workspace_bytes(*p, int(T));
  return QSFM_OK;
}

qsfm_status qsfm_lightning_indexer(const qsfm_indexer_params* pp, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  long long T = 0;
  const qsfm_status st = check_indexer(pp, &T);
  if (st != QSFM_OK) return st;
  const qsfm_indexer_params& p = *pp;
  if (T == 0) return QSFM_OK;
  if (p.query == nullptr || p.query_scale == nullptr || p.weights == nullptr || p.key == nullptr ||
      p.key_scale == nullptr || p.sparse_indices == nullptr)
    return QSFM_ERR_INVALID_ARG;
  if (p.layout_k == QSFM_LAYOUT_KV_PA_BBND && (p.block_table == nullptr || p.seqused_k == nullptr))
    return QSFM_ERR_INVALID_ARG;
  if (p.return_value && p.sparse_values == nullptr) return QSFM_ERR_INVALID_ARG;
  if (p.layout_k == QSFM_LAYOUT_KV_PA_BBND && (long long)p.num_blocks * p.block_size > kMaxPoolRows)
    return QSFM_ERR_UNSUPPORTED;
  if (!aligned(p.query, 16) || !aligned(p.key, 16) || !aligned(p.key_scale, 16)) return QSFM_ERR_INVALID_ARG;
  const void* words[] = {p.query_scale, p.weights, p.block_table, p.seqused_k, p.cmp_residual_k,
                         p.cu_seqlens_q, p.seqused_q, p.sparse_indices, p.sparse_values, p.cu_seqlens_k,
                         p.output_idx_offset};
  for (const void* w : words)
    if (!aligned(w, 4)) return QSFM_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, 16) ||
      workspace_bytes < qsfm::indexer_workspace_bytes(p, int(T)))
    return QSFM_ERR_WORKSPACE;
  int* fault = fault_ptr();
  if (fault == nullptr) return QSFM_ERR_CUDA;
  const NvtxRange range("qsfm_lightning_indexer");
  return cuda_status(qsfm::launch_indexer(p, int(T), workspace, fault, static_cast<cudaStream_t>(stream)));
}

qsfm_status qsfm_get_device_status(int32_t* fault_word) {
  if (fault_word == nullptr) return QSFM_ERR_INVALID_ARG;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fault_word, sizeof(int)) != cudaSuccess) return QSFM_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_fault_word, &zero, sizeof(int)) != cudaSuccess) return QSFM_ERR_CUDA;
  *fault_word = v;
  return v == 0 ? QSFM_OK : QSFM_ERR_DEVICE_FAULT;
}

const char* qsfm_status_string(qsfm_status s) {
  switch (s) {
    case QSFM_OK: return "ok";
    case QSFM_ERR_INVALID_ARG: return "invalid argument";
    case QSFM_ERR_UNSUPPORTED: return "unsupported shape or option";
    case QSFM_ERR_CUDA: return "CUDA runtime error";
    case QSFM_ERR_WORKSPACE: return "workspace missing or too small";
    case QSFM_ERR_DEVICE_FAULT: return "device fault word set";
    case QSFM_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

int32_t qsfm_abi_version(void) { return QSFM_ABI_VERSION; }

int32_t qsfm_last_cuda_error(const char** name) {
  const int e = g_last_cuda_error;
  if (name != nullptr) *name = e != 0 ? cudaGetErrorName(cudaError_t(e)) : "cudaSuccess";
  return e;
}

}  // extern "C"
