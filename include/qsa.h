/*
 * qsa.h -- C ABI of the QSA (Qwen4Exp learned sparse attention) layer step
 * for NVIDIA GB300 (sm_103a).
 *
 * One layer step runs four stages over a batch of query rows:
 *   1. compress  -- indexer query prep (Gemma RMSNorm, NeoX RoPE / interleaved
 *                   MRoPE, cast), group pooling into the compressed-key cache
 *                   and the raw-key ring commit;
 *   2. logits    -- index scores of each row against its visible compressed
 *                   keys;
 *   3. top-k     -- causal, per-request block top-k, expanded into the packed
 *                   selection buffer;
 *   4. sparse GQA-- paged grouped-query attention over the selected tokens,
 *                   with the sigmoid output gate.
 * Around them: the main-attention prepare (qsa_main_prepare, or fused into
 * stage 1 through qsa_step_args.main), the k-step MTP draft whose later
 * steps reuse step 0's selection (qsa_mtp_steps), the fused qkv + indexer
 * projection GEMM that produces the step's inputs (qsa_qkv_index_proj), and
 * stage 4 for callers that cannot give it a workspace
 * (qsa_sparse_gqa_noalloc).
 *
 * Sources: "vllm.models.qwen4_exp.nvidia.qsa" (QSAIndexer.forward and its
 * unfused reference path, Qwen4ExpQSAImpl.forward), "vllm.models.qwen4_exp.
 * nvidia.ops.qsa" (qsa_compress_groups_with_ratio, qsa_sparse_paged_attention,
 * qsa_store_cache_rows), "indexer_qsa.py" (apply_qsa_rope,
 * _supports_fused_pre_indexer) and the "FP8 E4M3 KV reader for QSA" patch
 * (_qsa_sparse_paged_gqa_splitk_kernel).
 *
 * Conventions shared by every entry point:
 *  - Every tensor argument is a DEVICE pointer owned by the caller; the
 *    library never allocates device memory and never frees caller memory.
 *    Scratch space is passed in as `ws` / `ws_bytes`, sized with
 *    qsa_workspace_bytes().
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL means the
 *    legacy default stream) and performs no host synchronisation and no
 *    device-to-host copy.
 *  - Host-side validation runs first; on any error nothing is launched and
 *    the status says why.  Out-of-range page ids, slots or token indices
 *    that only the device can see are masked (never dereferenced) and
 *    counted in a device error word that qsa_check_errors() reads.
 *  - Element types: "bf16" is IEEE bfloat16 stored as uint16; "e4m3" is
 *    OCP FP8 E4M3FN stored as one byte per element.
 *  - All index metadata is int32 unless stated; positions and slots are
 *    int64, as on the pages.
 *  - rows == 0 is a no-op that returns QSA_OK.
 */
#ifndef QSA_H
#define QSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum qsa_status {
  QSA_OK = 0,
  QSA_ERR_INVALID_ARG = 1,  /* null pointer or inconsistent argument */
  QSA_ERR_SHAPE = 2,        /* sizes do not fit together */
  QSA_ERR_DTYPE = 3,        /* unsupported element type */
  QSA_ERR_UNSUPPORTED = 4,  /* a configuration this build does not run */
  QSA_ERR_WORKSPACE = 5,    /* ws too small or misaligned */
  QSA_ERR_CUDA = 6,         /* a CUDA runtime / launch error */
  QSA_ERR_DEVICE_FAULT = 7  /* device-side masked out-of-range accesses */
} qsa_status;

enum { QSA_DTYPE_BF16 = 0, QSA_DTYPE_E4M3 = 1 };

/* Indexer configuration ("vllm.models.qwen4_exp.nvidia.qsa", QSAIndexer.__init__:
 * indexer_n_heads, indexer_head_dim, indexer_budget, indexer_compress_ratio,
 * rms_norm_eps, the indexer KV dtype; "indexer_qsa.py",
 * _supports_fused_pre_indexer: NeoX, head_dim 128, rotary_dim 64, one
 * indexer KV head, compress_ratio a power of two > 1, MRoPE as three
 * interleaved sections summing to rotary_dim / 2). */
typedef struct qsa_cfg {
  int32_t n_heads;          /* H_i, indexer query heads: 8, 16, 32 or 64 */
  int32_t head_dim;         /* D: must be 128 */
  int32_t rotary_dim;       /* must be 64 */
  int32_t compress_ratio;   /* r: power of two, 2..64 */
  int32_t token_topk;       /* K: multiple of r; K / r blocks are selected */
  float eps;                /* RMSNorm epsilon */
  int32_t index_dtype;      /* QSA_DTYPE_BF16 or QSA_DTYPE_E4M3 */
  int32_t mrope_section[3]; /* all 0: 1-D RoPE; else T,H,W sections, sum 32 */
  int32_t state_size;       /* S: compressor-state ring slots, >= r */
  int32_t cpage;            /* compressed keys per compressed-cache page */
  int32_t max_position;     /* rows of the cos/sin table */
} qsa_cfg;

/* Main attention configuration ("vllm.models.qwen4_exp.nvidia.qsa",
 * Qwen4ExpQSAImpl: num_heads, head_size, num_kv_heads; paged KV block size a
 * multiple of 16). */
typedef struct qsa_gqa_cfg {
  int32_t num_q_heads;   /* Hq, a multiple of Hkv; the group Hq / Hkv is 1..8 or 16
                            (other groups: QSA_ERR_UNSUPPORTED) */
  int32_t num_kv_heads;  /* Hkv */
  int32_t head_dim;      /* must be 128 */
  int32_t page_size;     /* tokens per KV block, a multiple of 16 */
  int32_t num_blocks;    /* KV blocks in the cache */
  /* KV cache element type ("0002-qwen4_exp-FP8-E4M3-KV-reader-for-QSA..."
   * patch; Qwen4ExpQSABackend.supported_kv_cache_dtypes "fp8_e4m3"):
   * QSA_DTYPE_BF16 (0, scales unused) or QSA_DTYPE_E4M3 (1): the cache holds
   * e4m3(x / scale) per tensor, and the reader folds k_scale into the scores
   * and v_scale into the normalised output.  e4m3 needs finite scales > 0. */
  int32_t kv_dtype;
  float k_scale;
  float v_scale;
} qsa_gqa_cfg;

/*
 * qsa_compress -- stage 1.
 * Follows "vllm.models.qwen4_exp.nvidia.qsa", QSAIndexer.forward, unfused
 * reference path (gemma_rmsnorm(q) -> apply_qsa_rope -> cast;
 * qsa_compress_groups_with_ratio -> gemma_rmsnorm(pooled) -> RoPE at the
 * group's first position -> cast -> qsa_store_cache_rows for compressed keys,
 * raw keys and rope positions) and "vllm.models.qwen4_exp.nvidia.ops.qsa",
 * qsa_compress_groups_with_ratio (argument shapes and checks).
 *
 *  projected_q  [rows, n_heads*D] bf16, row-contiguous; NULL skips query prep
 *  q_idx        [rows, n_heads, D] index dtype (output); NULL iff projected_q is
 *  raw_keys     [rows, 1, D] bf16
 *  positions    [rows, 1, 3] int64 (T, H, W; 1-D RoPE reads component 0)
 *  cos_sin      [max_position, rotary_dim] fp32: cos in the first half,
 *               sin in the second
 *  q_norm_w, k_norm_w  [D] bf16 (Gemma form: scale is 1 + w)
 *  ring         [ring_blocks, S, 1, D] bf16 compressor-state ring (in/out)
 *  ring_pos     [ring_blocks, S, 1, 3] int64 (in/out); required with MRoPE,
 *               must be NULL without it
 *  ring_block_table [reqs, ring_bt_stride] int32; column 0 is the request's ring
 *  token_to_req [rows], query_start_loc [reqs + 1], logical_positions [rows]
 *               (0-based position of the row's token in its request; the
 *               rows of a request are contiguous and consecutive)
 *  ccache       [cpages, cpage, 1, D] index dtype compressed-key cache (out)
 *  compressed_slots [rows] int64: flat slot (page * cpage + offset) where
 *               the group completed by this row is stored, < 0 for none.
 *               A row with a slot pools the r tokens ending at its position.
 * Ring slot of token t of request q: ring_block_table[q, 0] * S + t % S.  All
 * pooling reads see the ring as it was before the call; afterwards the ring
 * holds the newest S raw keys of each request.
 */
qsa_status qsa_compress(const qsa_cfg* cfg, const void* projected_q, void* q_idx,
                        const void* raw_keys, const int64_t* positions,
                        const float* cos_sin, const void* q_norm_w,
                        const void* k_norm_w, void* ring, int32_t ring_blocks,
                        int64_t* ring_pos, const int32_t* ring_block_table,
                        int32_t ring_bt_stride, const int32_t* token_to_req,
                        const int32_t* query_start_loc,
                        const int32_t* logical_positions, void* ccache,
                        int32_t cpages, const int64_t* compressed_slots,
                        int32_t rows, int32_t reqs, void* stream);

/*
 * qsa_index_logits -- stage 2.
 * Follows "vllm.models.qwen4_exp.nvidia.qsa", QSAIndexer.forward
 * (qsa_select_paged_decode / qsa_select_paged_prefill score the indexer
 * query against the paged compressed-key cache through its block table; the
 * selection is weight-free).  Score of row i and compressed key c < V(p_i),
 * V(p) = floor((p + 1) / r):
 *     logits[i, c] = (1 / (n_heads * sqrt(D))) * sum_h max(0, q_idx[i,h] . k_c)
 * with exact products and fp32 accumulation (tcgen05 MMA).
 *  q_idx        [rows, n_heads, D] index dtype
 *  ccache       [cpages, cpage, 1, D] index dtype
 *  cblock_table [reqs, cbt_stride] int32: key c of request q is at page
 *               cblock_table[q, c / cpage], offset c % cpage
 *  logits       [rows, ld] fp32 (out); entries c >= V(p_i) are not written
 *  max_visible  upper bound of V(p) over the rows (ld >= max_visible)
 *  ws, ws_bytes unused by this build (may be NULL / 0)
 */
qsa_status qsa_index_logits(const qsa_cfg* cfg, const void* q_idx,
                            const void* ccache, int32_t cpages,
                            const int32_t* cblock_table, int32_t cbt_stride,
                            const int32_t* token_to_req,
                            const int32_t* query_start_loc,
                            const int32_t* logical_positions, float* logits,
                            int64_t ld, int32_t max_visible, int32_t rows,
                            int32_t reqs, void* ws, size_t ws_bytes,
                            void* stream);

/*
 * qsa_topk -- stage 3 (block top-k and expand).
 * Follows "vllm.models.qwen4_exp.nvidia.qsa", QSAIndexer.forward
 * (block_indices of token_topk / compress_ratio columns, then
 * expand_qsa_block_indices) and the packed_output_width docstring.
 * For each row with V = V(p) visible blocks: the K_b = token_topk / r blocks
 * with the highest logits (ties to the lower block; all blocks if V <= K_b),
 * expanded in ascending order into their r tokens each, followed by the tail
 * tokens V*r .. p.  packed[i, 0 .. W-1] holds request-relative token indices
 * padded with -1; packed[i, W] holds their count, W = token_topk + r - 1.
 *  logits [rows, ld] fp32 (read only where c < V)
 *  packed [rows, W + 1] int32 (out)
 */
qsa_status qsa_topk(const qsa_cfg* cfg, const float* logits, int64_t ld,
                    int32_t max_visible, const int32_t* logical_positions,
                    int32_t* packed, int32_t rows, void* stream);

/*
 * qsa_sparse_gqa -- stage 4.
 * Follows "vllm.models.qwen4_exp.nvidia.ops.qsa", qsa_sparse_paged_attention
 * and the patch's _qsa_sparse_paged_gqa_splitk_kernel: for row i and query
 * head h (KV head h / (Hq / Hkv)), attention with scale D^-1/2 over the
 * packed[i, 0 .. n-1] tokens (n = packed[i, packed_width - 1]), zero when
 * n == 0, split-KV partials in fp32 merged by log-sum-exp, then
 * out = bf16(bf16(attn) * sigmoid(gate)) (or bf16(attn) when gate is NULL).
 *  q      [rows, Hq, D] bf16
 *  kv     [num_blocks, Hkv, page_size, 2*D] in the cfg's kv_dtype (bf16, or e4m3
 *         bytes), K in [..., :D], V in [..., D:]
 *  block_table [reqs, bt_stride] int32: token t of request q is in block
 *         block_table[q, t / page_size], offset t % page_size
 *  packed [rows, packed_width] int32; token_to_req [rows]
 *  gate   [rows, Hq, D] bf16 or NULL;  out [rows, Hq, D] bf16
 *  (query head h of a row reads KV head h / (Hq / Hkv))
 *  ws     scratch (split-KV partials and their merge tickets),
 *         qsa_workspace_bytes() bytes
 */
qsa_status qsa_sparse_gqa(const qsa_gqa_cfg* gcfg, const void* q, const void* kv,
                          const int32_t* block_table, int32_t bt_stride,
                          const int32_t* packed, int32_t packed_width,
                          const int32_t* token_to_req, const void* gate,
                          void* out, int32_t rows, void* ws, size_t ws_bytes,
                          void* stream);

/*
 * qsa_sparse_gqa_noalloc -- qsa_sparse_gqa for callers that cannot allocate.
 * No counterpart on the pages the method comes from: this is a library
 * convenience.  Some callers may not allocate device memory where attention
 * runs (an allocator frozen after start-up, a memory pool owned by someone
 * else, a plugin host that hands over only the call's tensors), so they
 * cannot provide the workspace qsa_sparse_gqa wants.  This variant keeps its
 * split-KV scratch in a static device array inside the library:
 * QSA_NOALLOC_SCRATCH_BYTES on every GPU that loads the library, held until
 * the process exits.  Arguments and results are those of qsa_sparse_gqa
 * without ws / ws_bytes; it allocates nothing.
 *  - Sizes whose split-KV partials need more than QSA_NOALLOC_SCRATCH_BYTES
 *    are rejected with QSA_ERR_WORKSPACE before anything is launched.
 *  - All calls on a device share the one array, which keeps the last call's
 *    contents (nothing in it has to start at zero).  Calls that can overlap
 *    on the GPU race on it: order them on one stream or with events.
 *  - The first call on each device looks up the array's device address with
 *    that device current and caches it; make that first call before any
 *    stream capture.  cudaDeviceReset unloads the library's device code and
 *    leaves that cached address stale: after resetting a device, do not call
 *    this entry point on it again in the same process.
 *  - Configuration checks are those of qsa_sparse_gqa.
 */
#define QSA_NOALLOC_SCRATCH_BYTES (4u << 20)
qsa_status qsa_sparse_gqa_noalloc(const qsa_gqa_cfg* gcfg, const void* q, const void* kv,
                                  const int32_t* block_table, int32_t bt_stride,
                                  const int32_t* packed, int32_t packed_width,
                                  const int32_t* token_to_req, const void* gate, void* out,
                                  int32_t rows, void* stream);

/*
 * Main-attention prepare, fused into the stage-1 launch of a layer step
 * ("vllm.models.qwen4_exp.nvidia.qsa", QSAIndexer.forward: the qsa_prepare
 * call with main_qkv, main_q_norm_weight, main_k_norm_weight, main_eps,
 * main_kv_cache, main_slot_mapping, main_k_scale, main_v_scale;
 * Qwen4ExpQSAAttention.__init__: the sigmoid output gate packed next to each
 * query head, q_norm / k_norm = GemmaRMSNorm(head_dim), the rotary embedding
 * shared with the indexer; Qwen4ExpQSAImpl.do_kv_cache_update: the K/V write
 * at slot_mapping).  Per row: q = RoPE(GemmaRMSNorm(q)) rounded to bf16, the
 * gate passed through (stage 4 applies the sigmoid), k = RoPE(GemmaRMSNorm(k))
 * and v written into the main KV cache at the row's slot (bf16, or
 * e4m3(x / scale) with the gcfg's scales), at the positions and with the
 * cos/sin table and MRoPE sections of the indexer.
 *  qkv          [rows, (2*Hq + 2*Hkv) * D] bf16: per query head [q | gate],
 *               then the Hkv K heads, then the Hkv V heads
 *  q_norm_w, k_norm_w  [D] bf16 (scale 1 + w); eps their epsilon
 *  q_out, gate_out     [rows, Hq, D] bf16 (out)
 *  kv           the main KV cache [num_blocks, Hkv, page, 2*D] (written)
 *  slot_mapping [rows] int64: block * page + offset of the row's token;
 *               < 0 writes nothing for that row
 */
typedef struct qsa_main_prep {
  const void* qkv;
  const void* q_norm_w;
  const void* k_norm_w;
  float eps;
  void* q_out;
  void* gate_out;
  void* kv;
  const int64_t* slot_mapping;
} qsa_main_prep;

/* The main-attention prepare alone (one launch), for callers that run the
 * stages one by one.  positions [rows, 1, 3] int64 and cos_sin as for
 * qsa_compress. */
qsa_status qsa_main_prepare(const qsa_cfg* cfg, const qsa_gqa_cfg* gcfg, const qsa_main_prep* m,
                            const int64_t* positions, const float* cos_sin, int32_t rows,
                            void* stream);

/*
 * qsa_qkv_index_proj -- the fused projection that feeds the layer step: one
 * GEMM y = x . w^T (bf16 inputs, fp32 accumulation on the tensor cores, one
 * bf16 rounding) over the stacked weights of the main attention and the
 * indexer, written as three row-major outputs.  Follows
 * "vllm.models.qwen4_exp.nvidia.qsa", Qwen4ExpQSAQKVIndexerLinear (the
 * indexer's index_qk_proj packed as shard 3 of the qkv GEMM),
 * Qwen4ExpQSAAttention.forward (qkv, projected_qk = qkv.split([2 q_size +
 * 2 kv_size, index_qk_size])) and QSAIndexer.forward (projected_q, raw_keys
 * = projected_qk.split((index_n_heads D, index_kv_heads D))).
 *  x            [rows, hidden] bf16, 16-byte aligned; hidden a multiple of 64
 *  w            [qkv_cols + index_q_cols + index_k_cols, hidden] bf16, 16-byte
 *               aligned: the main qkv weights (per query head [q | gate],
 *               then K, then V heads), then the indexer's query heads, then
 *               its key head
 *  qkv_out      [rows, qkv_cols] bf16 (the layer step's main qkv rows)
 *  index_q_out  [rows, index_q_cols] bf16 (projected_q)
 *  index_k_out  [rows, index_k_cols] bf16 (raw_keys)
 * An output may be NULL when its column count is 0.
 */
qsa_status qsa_qkv_index_proj(const void* x, const void* w, int32_t rows, int32_t hidden,
                              int32_t qkv_cols, int32_t index_q_cols, int32_t index_k_cols,
                              void* qkv_out, void* index_q_out, void* index_k_out, void* stream);

/* Arguments of one fused layer step (all device pointers; meanings as in the
 * stage calls above). */
typedef struct qsa_step_args {
  int32_t rows, reqs;
  int32_t max_visible;              /* upper bound of V(p) over the rows */
  const void* projected_q;          /* [rows, n_heads*D] bf16 */
  const void* raw_keys;             /* [rows, 1, D] bf16 */
  const int64_t* positions;         /* [rows, 1, 3] int64 */
  const float* cos_sin;             /* [max_position, rotary_dim] fp32 */
  const void* q_norm_w;             /* [D] bf16 */
  const void* k_norm_w;             /* [D] bf16 */
  void* ring;                       /* [ring_blocks, S, 1, D] bf16 */
  int32_t ring_blocks;
  int64_t* ring_pos;                /* [ring_blocks, S, 1, 3] or NULL */
  const int32_t* ring_block_table;  /* [reqs, ring_bt_stride] */
  int32_t ring_bt_stride;
  void* ccache;                     /* [cpages, cpage, 1, D] index dtype */
  int32_t cpages;
  const int32_t* cblock_table;      /* [reqs, cbt_stride] */
  int32_t cbt_stride;
  const int64_t* compressed_slots;  /* [rows] */
  const int32_t* token_to_req;      /* [rows] */
  const int32_t* query_start_loc;   /* [reqs + 1] */
  const int32_t* logical_positions; /* [rows] */
  int32_t* packed;                  /* [rows, token_topk + r] (out, or in with skip_topk) */
  const void* q;                    /* [rows, Hq, D] bf16 */
  const void* kv;                   /* [num_blocks, Hkv, page, 2D] bf16 or e4m3 */
  const int32_t* block_table;       /* [reqs, bt_stride] */
  int32_t bt_stride;
  const void* gate;                 /* [rows, Hq, D] bf16 or NULL */
  void* out;                        /* [rows, Hq, D] bf16 */
  /* NULL, or the main-attention prepare to fuse into stage 1: its q_out and
   * gate_out then feed stage 4 (q and gate above are ignored) and its kv must
   * be this step's kv. */
  const qsa_main_prep* main;
} qsa_step_args;

/*
 * qsa_layer_step -- stages 1 to 4 in order on one stream (with args->main,
 * stage 1 also prepares the main attention's q, gate and K/V cache rows).
 * Follows "vllm.models.qwen4_exp.nvidia.qsa", Qwen4ExpQSAAttention._run_qsa
 * and QSAIndexer.forward.  With skip_topk != 0 (MTP steps after step 0,
 * QSAIndexer.skip_topk) stage 1 still updates the ring and the compressed
 * cache, stages 2-3 are skipped and stage 4 reads the packed buffer as
 * given; skip_topk with a NULL packed buffer is QSA_ERR_INVALID_ARG ("QSA
 * top-k reuse requires an output buffer").
 */
qsa_status qsa_layer_step(const qsa_cfg* cfg, const qsa_gqa_cfg* gcfg,
                          const qsa_step_args* args, int32_t skip_topk,
                          void* ws, size_t ws_bytes, void* stream);

/*
 * qsa_mtp_steps -- the k layer steps of one multi-token-prediction draft, in
 * order on one stream: steps[0] selects (stages 1-4, writing the packed
 * buffer), steps[1 .. k-1] reuse that packed buffer unchanged (skip_topk:
 * stage 1 still writes the ring and the compressed cache, stage 4 attends
 * over the frozen selection).  Follows "vllm.models.qwen4_exp.nvidia.qsa",
 * QSAIndexer.skip_topk (top-k computed at the first MTP step, reused by the
 * later ones while the indexer cache keeps being updated) and the
 * topk_indices_buffer shared across the steps.
 *  steps  [k] step arguments; every step has the same rows, reqs and packed
 *         pointer (the persistent selection buffer) and its own per-step
 *         inputs and outputs (raw keys, positions, q, gate, out, ...)
 *  k      1 .. QSA_MTP_MAX_STEPS
 *  ws     one workspace of qsa_workspace_bytes() for these sizes, reused by
 *         every step (the steps run in stream order)
 * All k steps are validated before the first launch; on any error nothing is
 * launched.  No host synchronisation: the whole draft can be captured into
 * one CUDA graph.
 */
#define QSA_MTP_MAX_STEPS 16
qsa_status qsa_mtp_steps(const qsa_cfg* cfg, const qsa_gqa_cfg* gcfg, const qsa_step_args* steps,
                         int32_t k, void* ws, size_t ws_bytes, void* stream);

/* Scratch bytes needed by qsa_layer_step (and enough for every stage call)
 * for `rows` rows, `reqs` requests and V(p) <= max_visible.  The workspace
 * must be 256-byte aligned.  Returns 0 for invalid configurations. */
size_t qsa_workspace_bytes(const qsa_cfg* cfg, const qsa_gqa_cfg* gcfg,
                           int32_t rows, int32_t reqs, int32_t max_visible);

/* Number of kernel launches one qsa_layer_step call makes for these sizes:
 * 4 (compress, logits, top-k with the ring commit, sparse GQA with its split
 * merge), or 3 with skip_topk (compress, ring commit, sparse GQA).  0 if
 * invalid.  All but the first use programmatic dependent launch. */
int32_t qsa_step_launches(const qsa_cfg* cfg, const qsa_gqa_cfg* gcfg, int32_t rows,
                          int32_t reqs, int32_t skip_topk);

/* Split-KV factor qsa_sparse_gqa uses for `rows` rows (1 = no split, no
 * scratch).  0 if invalid. */
int32_t qsa_gqa_splits(const qsa_gqa_cfg* gcfg, int32_t rows, int32_t packed_width);

/* Static description of a status code. */
const char* qsa_status_string(qsa_status status);

/* Synchronises the current device, reads and clears the device error word
 * (count of masked out-of-range pages, slots or tokens since the last
 * call, and whether a bounded device-side wait gave up).  Returns
 * QSA_ERR_DEVICE_FAULT when it was non-zero, QSA_ERR_CUDA on a CUDA error,
 * else QSA_OK.  `count` may be NULL. */
qsa_status qsa_check_errors(int64_t* count);

/* Library version string. */
const char* qsa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* QSA_H */
