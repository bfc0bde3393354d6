/*
 * qsfm.h — C ABI of the quantized shared-KV sparse MLA attention forward
 * (QuantSparseFlashMla / KvQuantSparseAttnSharedKv) for sm_103a.
 *
 * What is computed (QuantSparseFlashMla, "功能说明" (function description),
 * formula O = softmax(Q K~^T * softmax_scale) V~ with K~ = V~; the per-head
 * sink is the "sinks" row of its "参数说明" (parameter) table):
 *
 *   for every query token t (batch b, position s) and head h (N1 = 64 or
 *   128 heads, D = 512, one latent KV head, N2 = 1):
 *     rows(t) = ori rows inside the band / causal window of t
 *             ++ cmp rows (CSA: the valid entries of cmp_sparse_indices[t];
 *                          HCA: every causally visible compressed row)
 *     K~[j, d] = e4m3fn(kv[j, d]) * scale[j, d / 64]
 *     x_j      = softmax_scale * sum_d Q[t, h, d] K~[j, d]
 *     O[t, h]  = sum_j e^{x_j} K~[j, :] / (sum_j e^{x_j} + e^{sink_h})
 *     lse[t,h] = log sum_j e^{x_j}          (the sink is not included)
 *   A token with no attended row gets O = 0 and lse = -inf.
 *
 * Modes (QuantSparseFlashMla, "约束说明" (constraints), third bullet):
 *   SWA  cmp_kv == NULL                        ori window only
 *   CSA  cmp_kv != NULL, cmp_sparse_indices    window + top-k compressed rows
 *   HCA  cmp_kv != NULL, indices == NULL       window + all visible cmp rows
 *
 * Data layout (all device memory is owned by the caller; the library never
 * allocates, frees or keeps pointers after a call returns):
 *   q            bf16  BSND [B, S1, N1, 512] or TND [T1, N1, 512]
 *   attn_out     bf16  same shape as q
 *   softmax_lse  fp32  BSND [B, 1, S1, N1] / TND [1, T1, N1]
 *                      (KvQuantSparseAttnSharedKv, parameter table, row
 *                      softmax_lse); element (token t, head h) at t*N1 + h
 *   ori_kv       fp8 e4m3fn, paged [ori_num_blocks, 128, 1, 512]
 *   cmp_kv       fp8 e4m3fn, paged [cmp_num_blocks, 128, 1, 512]
 *   ori_scale / cmp_scale
 *                fp32 [num_blocks, 128, 1, 8]: one dequant scale per
 *                64-element tile of a row, paged exactly like its KV
 *                (KvQuantSparseAttnSharedKv, parameter table, rows
 *                kv_quant_mode and tile_size: per-tile quantisation, tile 64)
 *   *_block_table int32 [B, *_max_blocks]: logical block -> physical block
 *                (QuantSparseFlashMla, "约束说明", PageAttention bullets)
 *   non-paged KV (layout_kv BSND / TND, QuantSparseFlashMla "约束说明" on
 *   layout_kv): ori_kv [B, S2, 1, row] / [T2, 1, row] and cmp_kv
 *                [B, S3, 1, row] / [T3, 1, row], scales [.., 8] alike;
 *                batch b's row j is at [b, j] (BSND) or at
 *                cu_seqlens_ori_kv[b] + j / cu_seqlens_cmp_kv[b] + j (TND);
 *                no block tables
 *   ori_sparse_indices int32 BSND [B, S1, 1, K1] / TND [T1, 1, K1] or NULL:
 *                discrete picks of ori rows (a logical ori row of the
 *                token's batch; -1 = invalid). When given they replace the
 *                contiguous ori range: the token attends the entries (the
 *                first ori_topk_length[t] when that is given) that lie in
 *                its ori mask range, each occurrence once, in index order
 *   cmp_sparse_indices int32 BSND [B, S1, 1, K2] / TND [T1, 1, K2];
 *                an entry is a logical compressed-row index of the token's
 *                own batch; -1 (or any value outside the visible range) is
 *                ignored
 *   cu_seqlens_q int32 [B + 1], prefix sums from 0 (required for TND)
 *   seqused_q    int32 [B] or NULL (BSND: rows s >= seqused_q[b] are
 *                padding; they get O = 0, lse = -inf)
 *   seqused_ori_kv int32 [B]: ori length S2 of each batch. Required for
 *                paged KV; optional for BSND KV (default: the S2
 *                dimension); must be NULL for TND KV (S2 = cu_seqlens_ori_kv
 *                difference)
 *   seqused_cmp_kv int32 [B] or NULL (default: floor(S2 / cmp_ratio) for
 *                paged KV, the S3 dimension for BSND KV, the
 *                cu_seqlens_cmp_kv difference for TND KV)
 *   cmp_residual_kv int32 [B] or NULL (default 0), 0 <= r_b < cmp_ratio
 *   cmp_topk_length int32 [T] or NULL: only the first n entries of the
 *                token's index row are read
 *   sinks        fp32 [N1] or NULL (NULL: no sink)
 *   metadata     int32 [1024] written by qsfm_metadata()
 *
 * Query position alignment is bottom-right: p = S2 - S1_b + s on the ori
 * side and p_c = cmp_len * cmp_ratio + residual - S1_b + s on the cmp side.
 * ori mask mode 4 (band) keeps rows max(0, p - wl) .. min(S2 - 1, p + wr),
 * -1 meaning no bound on that side; mode 3 keeps rows <= p; mode 0 keeps all.
 * cmp mask mode 3 keeps compressed rows c < floor((p_c + 1) / cmp_ratio)
 * (clipped to [0, cmp_len]); mode 0 keeps all cmp_len rows.
 *
 * Every call is asynchronous on the given stream and never reads device
 * memory back to the host, so the calls may be captured in a CUDA graph
 * (QuantSparseFlashMla, "约束说明": aclgraph mode). Argument errors are found
 * on the host before anything is launched and are returned as status codes.
 * Bad device data (a block id outside the pool, a block-table column past
 * its width) is not trapped: the row is skipped and a bit is set in the
 * device fault word, which qsfm_get_device_status() reads.
 */
#ifndef QSFM_H
#define QSFM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QSFM_ABI_VERSION 6
#define QSFM_NUM_HEADS 64
#define QSFM_HEAD_DIM 512
#define QSFM_BLOCK_SIZE 128
#define QSFM_SCALES_PER_ROW 8
#define QSFM_METADATA_INTS 1024
#define QSFM_MAX_CTAS 256
#define QSFM_PACKED_ROW_BYTES 640
#define QSFM_BF16_ROW_BYTES 1024

/* KV row formats (qsfm_params.kv_layout). */
typedef enum {
  /* fp8 e4m3fn rows [blocks, 128, 1, 512] with fp32 scale tensors
   * [blocks, 128, 1, 8], one scale per 64 elements (the default). */
  QSFM_KV_FP8_FP32_SCALES = 0,
  /* Packed 640-byte rows [blocks, 128, 1, 640] (KvQuantSparseAttnSharedKv
   * constraints): bf16 rope (64 elements, bytes 0..127), e4m3fn nope (448
   * elements, bytes 128..575), e8m0 scales (7, one per 64 nope elements,
   * bytes 576..582), zero padding to 640. The 512 elements of a row are
   * rope then nope; ori_scale and cmp_scale must be NULL. */
  QSFM_KV_PACKED640 = 1,
  /* bf16 rows [blocks, 128, 1, 512] without quantisation (the KV of
   * SparseCompressedFlashAttention); ori_scale and cmp_scale must be NULL. */
  QSFM_KV_BF16 = 2
} qsfm_kv_layout;

typedef enum {
  QSFM_OK = 0,
  QSFM_ERR_INVALID_ARG = 1,  /* a constraint of the op is violated        */
  QSFM_ERR_UNSUPPORTED = 2,  /* valid for the op but not built             */
  QSFM_ERR_CUDA = 3,         /* a CUDA runtime call failed                */
  QSFM_ERR_WORKSPACE = 4,    /* workspace NULL or smaller than required   */
  QSFM_ERR_DEVICE_FAULT = 5, /* the device fault word is non-zero         */
  QSFM_ERR_TIMEOUT = 6       /* reserved for bounded device waits         */
} qsfm_status;

typedef enum { QSFM_LAYOUT_BSND = 0, QSFM_LAYOUT_TND = 1 } qsfm_q_layout;

/* KV storage (qsfm_params.layout_kv; QuantSparseFlashMla parameter table
 * row layout_kv and its constraints: BSND / TND KV only with the same q
 * layout, paged KV with either). */
typedef enum {
  QSFM_LAYOUT_KV_PA_BBND = 0, /* paged 128-row blocks through block tables  */
  QSFM_LAYOUT_KV_BSND = 1,    /* [B, S, 1, row] per batch slab              */
  QSFM_LAYOUT_KV_TND = 2      /* [T, 1, row], batches at cu_seqlens_*_kv    */
} qsfm_layout_kv;

/* Device fault word bits (qsfm_get_device_status). */
#define QSFM_FAULT_ORI_BLOCK_ID   0x1  /* ori block table entry outside pool */
#define QSFM_FAULT_CMP_BLOCK_ID   0x2  /* cmp block table entry outside pool */
#define QSFM_FAULT_ORI_TABLE_COL  0x4  /* ori row beyond the table width     */
#define QSFM_FAULT_CMP_TABLE_COL  0x8  /* cmp row beyond the table width     */
#define QSFM_FAULT_METADATA       0x10 /* metadata header does not match     */
#define QSFM_FAULT_TIMEOUT        0x20 /* a bounded device wait ran out      */
#define QSFM_FAULT_RANGE          0x40 /* an fp8 KV row dequantises past
                                          2^22: its values were clamped    */
#define QSFM_FAULT_KV_ROW         0x80 /* a non-paged KV row past the end of
                                          its tensor (skipped)             */

/*
 * All inputs, attributes and outputs of one forward call. Pointers are
 * device pointers; NULL marks an absent optional input. q, ori_kv, cmp_kv and
 * attn_out must be 16-byte aligned and every other pointer 4-byte aligned
 * (QSFM_ERR_INVALID_ARG otherwise). The parameter names follow
 * QuantSparseFlashMla, "参数说明" (parameter table).
 * Size limits of the kernels' 32-bit index arithmetic (QSFM_ERR_UNSUPPORTED
 * beyond them; every batch that fits in device memory is far below): at
 * most 2^24 work units (tokens x n1 / 64), k2 <= 65536, and fewer than 2^31
 * rows in each KV pool (num_blocks x block_size).
 */
typedef struct qsfm_params {
  /* shapes */
  int32_t batch;          /* B                                               */
  int32_t max_s1;         /* BSND: S1. TND: unused                           */
  int32_t total_t;        /* TND: T1 (= q.shape[0]). BSND: unused            */
  int32_t n1;             /* query heads: 64 or 128 (the pages allow both)   */
  int32_t d;              /* head dim; must be 512                           */
  int32_t k2;             /* index row length K2 (CSA); 0 otherwise          */
  int32_t ori_block_size; /* tokens per ori block; only 128 is built         */
  int32_t cmp_block_size; /* tokens per cmp block; only 128 is built         */
  int32_t ori_max_blocks; /* ori_block_table row width                       */
  int32_t cmp_max_blocks; /* cmp_block_table row width                       */
  int32_t ori_num_blocks; /* physical blocks in the ori pool                 */
  int32_t cmp_num_blocks; /* physical blocks in the cmp pool                 */
  int32_t num_ctas;       /* most CTAs the work is planned over; 0 = SM
                             count. The plan's units are the 64-head groups
                             of the tokens (U = T * n1 / 64). With U >=
                             num_ctas the plan uses ceil(U / ceil(U /
                             num_ctas)) CTAs, the fewest that keep the same
                             units per CTA                                  */
  /* inputs (device) */
  const void* q;
  const void* ori_kv;
  const float* ori_scale;
  const void* cmp_kv;
  const float* cmp_scale;
  const int32_t* cmp_sparse_indices;
  const int32_t* ori_block_table;
  const int32_t* cmp_block_table;
  const int32_t* cu_seqlens_q;
  const int32_t* seqused_q;
  const int32_t* seqused_ori_kv;
  const int32_t* seqused_cmp_kv;
  const int32_t* cmp_residual_kv;
  const int32_t* cmp_topk_length;
  const float* sinks;
  const int32_t* metadata;
  /* attributes */
  float softmax_scale;
  int32_t cmp_ratio;      /* 1..128; must be 1 when cmp_kv is NULL           */
  int32_t ori_mask_mode;  /* 0, 3 or 4                                       */
  int32_t cmp_mask_mode;  /* 0 or 3                                          */
  int32_t ori_win_left;   /* -1 or >= 0; >= 0 only with ori_mask_mode 4      */
  int32_t ori_win_right;  /* -1 or >= 0; >= 0 only with ori_mask_mode 4      */
  int32_t layout_q;       /* qsfm_q_layout                                   */
  int32_t return_lse;     /* non-zero: write softmax_lse                     */
  /* outputs (device) */
  void* attn_out;
  float* softmax_lse;
  /* appended in ABI version 2 */
  int32_t kv_layout;      /* qsfm_kv_layout of ori_kv and cmp_kv (both)      */
  /* appended in ABI version 3 */
  int32_t layout_kv;      /* qsfm_layout_kv of ori_kv and cmp_kv (both)      */
  int32_t ori_kv_len;     /* BSND / TND KV: length of ori_kv's sequence axis
                             (S2 of [B, S2, 1, row], T2 of [T2, 1, row])     */
  int32_t cmp_kv_len;     /* the same for cmp_kv (S3 / T3)                   */
  int32_t k1;             /* ori_sparse_indices row length K1; 0 without     */
  const int32_t* cu_seqlens_ori_kv;  /* int32 [B + 1]: TND KV (required)      */
  const int32_t* cu_seqlens_cmp_kv;  /* int32 [B + 1]: TND KV with cmp_kv    */
  const int32_t* ori_sparse_indices; /* see the data layout above            */
  const int32_t* ori_topk_length;    /* int32 [T] or NULL: entries of the
                                        token's ori index row that count    */
} qsfm_params;

/* Fill *p with the defaults of the op: n1 64, d 512, block size 128,
 * cmp_ratio 1, ori mask 4 with window 127/0 (KvQuantSparseAttnSharedKv,
 * parameter table rows ori_mask_mode, ori_win_left, ori_win_right), cmp mask
 * 3, softmax_scale 1/sqrt(512), layout BSND, all pointers NULL. */
void qsfm_params_init(qsfm_params* p);

/*
 * Plan the work of one forward call over p->num_ctas CTAs (the split-core
 * plan of QuantSparseFlashMlaMetadata, QuantSparseFlashMla "功能说明",
 * calling sequence steps 1-3). Reads cu_seqlens_q / seqused_* /
 * cmp_residual_kv / cmp_topk_length on the device and writes the int32[1024]
 * plan to metadata_out (device memory, caller-owned). Launches one small
 * kernel on `stream`; nothing is read back.
 * Errors: QSFM_ERR_INVALID_ARG for a NULL metadata_out or invalid params.
 */
qsfm_status qsfm_metadata(const qsfm_params* p, int32_t* metadata_out,
                          void* stream /* cudaStream_t */);

/* Bytes of device workspace qsfm_forward() needs for p (partial outputs of
 * work split across CTAs). May be 0. */
qsfm_status qsfm_forward_workspace_size(const qsfm_params* p, size_t* bytes);

/*
 * The forward pass: attention kernel, then (only when the plan may split a
 * token across CTAs) the log-sum-exp combine kernel. Writes attn_out and,
 * when return_lse is set, softmax_lse. p->metadata must come from
 * qsfm_metadata() with the same shapes and lengths (QuantSparseFlashMla,
 * "约束说明": metadata is required, shape [1024]).
 * workspace: device memory of at least qsfm_forward_workspace_size() bytes.
 */
qsfm_status qsfm_forward(const qsfm_params* p, void* workspace,
                         size_t workspace_bytes, void* stream);

/* The two stages of qsfm_forward(), callable separately (for timing). */
qsfm_status qsfm_attention(const qsfm_params* p, void* workspace,
                           size_t workspace_bytes, void* stream);
qsfm_status qsfm_combine(const qsfm_params* p, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * qsfm_forward() for callers that cannot allocate device memory. The paper
 * has no counterpart: this is an addition of this library.
 *
 * Some callers cannot call cudaMalloc: code that runs inside another
 * framework's memory pool, plugin hosts that hand over only the input and
 * output buffers, serving loops that forbid allocation once running. This
 * entry point allocates nothing. Instead of a workspace argument it uses a
 * fixed scratch array of QSFM_NOALLOC_SCRATCH_BYTES that the library
 * reserves in the memory of every GPU that loads it, held until the process
 * exits. The caller still passes all inputs and outputs (and the metadata
 * from qsfm_metadata()) in p.
 *   - Returns QSFM_ERR_WORKSPACE, launching nothing, when the plan needs
 *     more than QSFM_NOALLOC_SCRATCH_BYTES of partial results (that happens
 *     only when tokens may be split over CTAs, i.e. fewer query tokens than
 *     p->num_ctas; the need is 2 * num_ctas * 131328 bytes rounded up, so at
 *     most 31 CTAs fit). qsfm_forward_workspace_size() gives the need.
 *   - The first call on a device looks up the array's device address with
 *     that device current; make it before any stream capture.
 *   - All calls share the array, which keeps the last call's contents;
 *     nothing in it needs to start at zero. Calls that overlap on the GPU
 *     (other streams or threads) race on it.
 */
#define QSFM_NOALLOC_SCRATCH_BYTES (8u << 20)
qsfm_status qsfm_forward_noalloc(const qsfm_params* p, void* stream);

/*
 * Debug export of the row resolution the attention kernel uses. For each
 * of the n query tokens in tokens[] (device int32), writes the token's row
 * slots in the kernel's order (ori window rows, then cmp slots), up to
 * max_rows of them:
 *   rows_out    uint8 [n, max_rows, R]    the bytes of the resolved row in
 *                                         the pool's own format, R = 512
 *                                         (fp8), 640 (packed) or 1024 (bf16)
 *   scales_out  fp32  [n, max_rows, 8]    its dequant scales (fp8 only)
 *   row_ids_out int32 [n, max_rows]       (source << 30) | logical row, with
 *                                         source 0 = ori, 1 = cmp; -1 for a
 *                                         slot that is masked out
 *   counts_out  int32 [n]                 number of slots of the token
 * Masked slots get zero bytes and zero scales. All buffers are device memory
 * and rows_out must be 16-byte aligned. rows_out and scales_out may both be
 * NULL: then only the row ids and counts are written. For the fp8 format
 * rows_out and scales_out are given together or not at all; for the others
 * scales_out must be NULL (QSFM_ERR_INVALID_ARG otherwise). row_ids_out is
 * required when max_rows > 0.
 */
qsfm_status qsfm_debug_gather(const qsfm_params* p, const int32_t* tokens,
                              int32_t n, int32_t max_rows, uint8_t* rows_out,
                              float* scales_out, int32_t* row_ids_out,
                              int32_t* counts_out, void* stream);

/*
 * Debug check of the bounded waits every kernel of the library uses (no GPU
 * fault, no hang). One block: a thread waits with a limit of timeout_ns on
 * an mbarrier that nothing arrives on; when the limit runs out it raises the
 * block's abort flag and sets QSFM_FAULT_TIMEOUT in the fault word. A thread
 * of another warp waits on a second such barrier with a limit 1000 times as
 * long and gives up as soon as it sees the abort flag. Writes the two waits'
 * durations in ns to elapsed_ns_out[0..1] (device memory, caller-owned).
 * Errors: QSFM_ERR_INVALID_ARG for a NULL output, or timeout_ns of 0 or
 * above one second.
 */
qsfm_status qsfm_debug_bounded_wait(uint64_t timeout_ns, uint64_t* elapsed_ns_out, void* stream);

/*
 * Lightning-indexer top-k (QuantLightningIndexerV2, "功能说明" formula and
 * "参数说明" (parameter table); quant mode 1: FLOAT8_e4m3fn query and key,
 * fp32 dequant scales and weights). For every query token t (batch b,
 * position s) and every key j it may see:
 *   score_j = sum_h weights[t, h] * ReLU(query_scale[t, h] * key_scale[j]
 *                                        * sum_d query[t, h, d] key[j, d])
 * and sparse_indices[t] lists the topk keys of largest score (the smaller
 * key index first among equal scores) in ascending key order, then -1 up
 * to topk (valid entries first, -1 after, as KvQuantSparseAttnSharedKv's
 * constraints want of an index row). Keys visible to the token: all
 * j < seqused_k[b] (mask_mode 0), or only j < floor((p_c + 1) / cmp_ratio)
 * with p_c = seqused_k[b] * cmp_ratio + cmp_residual_k[b] - S1_b + s
 * (mask_mode 3, the compressed rows' right-down-causal rule). A padded
 * query row (seqused_q) gets -1 everywhere.
 *
 * Layout (all device memory, caller-owned):
 *   query        e4m3fn bytes BSND [B, S1, heads, dim] / TND [T, heads, dim]
 *   query_scale  fp32 [T, heads];  weights fp32 [T, heads]
 *   key          e4m3fn bytes (parameter table: layout_k):
 *                  PA_BBND (default) paged [num_blocks, 128, 1, dim] through
 *                    block_table int32 [B, max_blocks], seqused_k[b] keys
 *                    (seqused_k required);
 *                  BSND [B, max_sk, 1, dim], batch b's key j at [b, j],
 *                    seqused_k[b] keys (max_sk when seqused_k is NULL);
 *                  TND [total_k, 1, dim], batch b's key j at row
 *                    cu_seqlens_k[b] + j, cu_seqlens_k[b + 1] - cu_seqlens_k[b]
 *                    keys (cu_seqlens_k int32 [B + 1] required, seqused_k
 *                    NULL)
 *   key_scale    fp32, the key's layout without the dim axis
 *   output_idx_offset int32 [B] or NULL: every valid index of a batch-b row
 *                is reported plus output_idx_offset[b] (-1 stays -1)
 *   cmp_residual_k int32 [B] or NULL (0);  cu_seqlens_q int32 [B + 1]
 *                (required for TND);  seqused_q int32 [B] or NULL: query
 *                rows of batch b from seqused_q[b] on are padding (all -1;
 *                the other rows keep their positions, S1_b being the chunk
 *                length of the layout), for BSND and TND alike
 *   sparse_indices int32 [T, 1, topk] (out)
 *   sparse_values  bf16 [T, 1, topk] (out, written when return_value != 0;
 *                the scores of the listed keys, -inf after them)
 * Built shapes (QSFM_ERR_UNSUPPORTED otherwise): dim = 128, 1 <= heads
 * <= 64, 1 <= topk <= 8192, block size 128, at most 2^20 query rows, at
 * most 32768 keys per batch and at most max_blocks * 128 (paged) or max_sk
 * (BSND) of them; a larger key count is cut and flagged
 * (QSFM_FAULT_KV_ROW past 32768 or past the end of a TND key tensor, else
 * QSFM_FAULT_CMP_TABLE_COL). A block id outside [0, num_blocks) is flagged
 * with QSFM_FAULT_CMP_BLOCK_ID, its keys score -inf and are not read.
 * Pointers: query, key, key_scale 16-byte aligned, the rest 4-byte aligned.
 */
typedef struct qsfm_indexer_params {
  int32_t batch;        /* B                                                */
  int32_t max_s1;       /* BSND: S1                                         */
  int32_t total_t;      /* TND: T (query rows)                              */
  int32_t heads;        /* g, query heads of the indexer                    */
  int32_t dim;          /* d, must be 128                                   */
  int32_t topk;         /* 1 .. 8192                                        */
  int32_t block_size;   /* keys per block; only 128 is built                */
  int32_t max_blocks;   /* block_table row width                            */
  int32_t num_blocks;   /* blocks in the key pool                           */
  int32_t layout_q;     /* qsfm_q_layout                                    */
  int32_t mask_mode;    /* 0 or 3                                           */
  int32_t cmp_ratio;    /* 1 .. 128                                         */
  int32_t return_value; /* non-zero: write sparse_values                    */
  const void* query;
  const float* query_scale;
  const float* weights;
  const void* key;
  const float* key_scale;
  const int32_t* block_table;
  const int32_t* seqused_k;
  const int32_t* cmp_residual_k;
  const int32_t* cu_seqlens_q;
  const int32_t* seqused_q;
  int32_t* sparse_indices;
  void* sparse_values;
  /* version 6: the key layouts and the index offset */
  int32_t layout_k;     /* qsfm_kv_layout: PA_BBND (default), BSND or TND   */
  int32_t max_sk;       /* BSND keys: S_k, the key tensor's S dimension     */
  int32_t total_k;      /* TND keys: T_k, the key tensor's rows             */
  const int32_t* cu_seqlens_k;
  const int32_t* output_idx_offset;
} qsfm_indexer_params;

/* Defaults: dim 128, heads 64, topk 2048 (the page's default), block size
 * 128, mask_mode 0, cmp_ratio 1, layout BSND, all pointers NULL. */
void qsfm_indexer_params_init(qsfm_indexer_params* p);

/* Bytes of device workspace qsfm_lightning_indexer() needs for p: one fp32
 * score row of min(32768, max_blocks * 128) entries per query row. Reads
 * no device memory. Errors as qsfm_lightning_indexer() for the attributes. */
qsfm_status qsfm_lightning_indexer_workspace_size(const qsfm_indexer_params* p, size_t* bytes);

/* The indexer's top-k: a score kernel writes every visible key's score into
 * the workspace, a select kernel then lists each row's top-k. workspace:
 * caller-owned device memory, 16-byte aligned, of at least
 * qsfm_lightning_indexer_workspace_size() bytes, not read before it is
 * written. Asynchronous on `stream`, no allocation, nothing read back.
 * Errors: QSFM_ERR_INVALID_ARG (missing or misaligned pointers, bad
 * attributes), QSFM_ERR_UNSUPPORTED (shapes not built), QSFM_ERR_WORKSPACE
 * (workspace NULL, misaligned or too small). */
qsfm_status qsfm_lightning_indexer(const qsfm_indexer_params* p, void* workspace, size_t workspace_bytes,
                                   void* stream);

/* Synchronously read and clear the device fault word of the current
 * device (QSFM_FAULT_* bits). Returns QSFM_ERR_DEVICE_FAULT when non-zero. */
qsfm_status qsfm_get_device_status(int32_t* fault_word);

const char* qsfm_status_string(qsfm_status s);
int32_t qsfm_abi_version(void);

/* The CUDA runtime error code behind the last QSFM_ERR_CUDA an entry point
 * returned on the calling host thread (0 if none), and its name in *name
 * when name is not NULL (a static string). Not cleared by later calls. */
int32_t qsfm_last_cuda_error(const char** name);

#ifdef __cplusplus
}
#endif

#endif /* QSFM_H */
