// C ABI of the QSA layer step (declared in include/qsa.h): host-side
// validation, workspace layout, TMA descriptor encoding and kernel launch
// order.  Nothing here allocates device memory.
#include <mutex>

#include "qsa.h"
#include "qsa_device.cuh"
#include "qsa_kernels.h"

namespace qsa {
namespace {

__device__ unsigned long long g_error_word;

constexpr int kMaxDevices = 64;
unsigned long long* g_err_ptr[kMaxDevices] = {};
std::mutex g_err_mu;

// Device address of the error word for the current device (resolved once per
// device with that device current).
unsigned long long* error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_err_mu);
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<unsigned long long*>(p);
  }
  return g_err_ptr[dev];
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D map over [outer, 128 elements] rows with a 128-byte-wide box of
// `box_rows` rows, 128-byte swizzle, zero fill out of bounds.
bool encode_rows_map(CUtensorMap* map, const void* base, int elem_bytes, long long outer,
                     int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const CUtensorMapDataType dt =
      elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(128 * elem_bytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elem_bytes), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Set while qsa_mtp_steps validates all of its steps before it launches any
// of them: the stage helpers then return right before their launches.
thread_local bool t_validate_only = false;

struct ValidateOnly {
  ValidateOnly() { t_validate_only = true; }
  ~ValidateOnly() { t_validate_only = false; }
};

// 2-D bf16 map over [outer, inner] row-major with a box of 64 elements x
// box_rows rows, 128-byte swizzle, zero fill out of bounds.
bool encode_bf16_2d(CUtensorMap* map, const void* base, long long inner, long long outer,
                    int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner * 2)};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool pow2(long long x) { return x > 0 && (x & (x - 1)) == 0; }
size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

qsa_status check_cfg(const qsa_cfg* c) {
  if (c == nullptr) return QSA_ERR_INVALID_ARG;
  if (c->head_dim != 128 || c->rotary_dim != 64) return QSA_ERR_UNSUPPORTED;
  if (!(c->n_heads == 8 || c->n_heads == 16 || c->n_heads == 32 || c->n_heads == 64))
    return QSA_ERR_UNSUPPORTED;
  if (!pow2(c->compress_ratio) || c->compress_ratio < 2 || c->compress_ratio > 64)
    return QSA_ERR_UNSUPPORTED;
  if (c->token_topk <= 0 || c->token_topk % c->compress_ratio != 0) return QSA_ERR_INVALID_ARG;
  if (!(c->eps >= 0.f)) return QSA_ERR_INVALID_ARG;
  if (c->index_dtype != QSA_DTYPE_BF16 && c->index_dtype != QSA_DTYPE_E4M3) return QSA_ERR_DTYPE;
  const int* s = c->mrope_section;
  const bool any = s[0] || s[1] || s[2];
  if (any && (s[0] < 0 || s[1] < 0 || s[2] < 0 || s[0] + s[1] + s[2] != 32))
    return QSA_ERR_UNSUPPORTED;
  if (c->state_size < c->compress_ratio) return QSA_ERR_SHAPE;
  if (!pow2(c->cpage) || c->cpage > 128) return QSA_ERR_UNSUPPORTED;
  if (c->max_position < 1) return QSA_ERR_INVALID_ARG;
  return QSA_OK;
}

int elem_bytes(const qsa_cfg* c) { return c->index_dtype == QSA_DTYPE_E4M3 ? 1 : 2; }

// Rows per logits row group and the padded MMA N it implies.
void logits_grouping(const qsa_cfg* c, int rows, int reqs, int* R, int* npad) {
  const int max_r = 256 / c->n_heads;
  int avg = reqs > 0 ? (rows + reqs - 1) / reqs : 1;
  int r = 1;
  while (r < avg && r < max_r) r <<= 1;
  if (r > max_r) r = max_r;
  int n = r * c->n_heads;
  int np = 32;
  while (np < n) np <<= 1;
  *R = r;
  *npad = np;
}

int max_groups_for(int rows, int reqs, int R) {
  long long a = static_cast<long long>(rows) / R + reqs;
  if (a > rows) a = rows;
  return static_cast<int>(a < 1 ? 1 : a);
}

long long logits_ld(int max_visible) { return (static_cast<long long>(max_visible) + 3) / 4 * 4; }

// The logits kernel needs no scratch (each CTA finds its own row group).
size_t logits_ws_bytes(int, int, const qsa_cfg*) { return 0; }

// GQA scratch: fp32 partial slots, their log-sum-exps and the merge tickets.
struct GqaLayout {
  int splits;
  size_t po, pl, tickets, total;  // byte offsets of the regions, total size
};

GqaLayout gqa_layout(const qsa_gqa_cfg* g, int rows, int packed_width) {
  GqaLayout L{};
  L.splits = gqa_num_splits(rows, g->num_kv_heads, packed_width, sm_count());
  if (L.splits == 1) return L;
  const long long slots = static_cast<long long>(L.splits) * rows * g->num_kv_heads;
  L.po = 0;
  const int group = g->num_q_heads / g->num_kv_heads;
  L.pl = align256(static_cast<size_t>(slots) * group * 128 * sizeof(float));
  L.tickets = L.pl + align256(static_cast<size_t>(slots) * group * sizeof(float));
  L.total = L.tickets + align256(static_cast<size_t>(rows) * g->num_kv_heads * sizeof(unsigned));
  return L;
}

size_t gqa_ws_bytes(const qsa_gqa_cfg* g, int rows, int packed_width) {
  return gqa_layout(g, rows, packed_width).total;
}

qsa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? QSA_OK : QSA_ERR_CUDA; }

size_t topk_limit_bytes() { return 220 * 1024; }

// Checks the main-attention prepare's arguments and adds them to p (whose
// positions, cos/sin table and RoPE layout it shares).
qsa_status fill_main(CompressParams* p, const qsa_gqa_cfg* g, const qsa_main_prep* m) {
  const qsa_status st = check_gcfg(g);
  if (st != QSA_OK) return st;
  if (!m->qkv || !m->q_norm_w || !m->k_norm_w || !m->q_out || !m->gate_out || !m->kv ||
      !m->slot_mapping)
    return QSA_ERR_INVALID_ARG;
  if (!(m->eps >= 0.f)) return QSA_ERR_INVALID_ARG;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(m->qkv) | reinterpret_cast<uintptr_t>(m->q_norm_w) |
                        reinterpret_cast<uintptr_t>(m->k_norm_w) | reinterpret_cast<uintptr_t>(m->q_out) |
                        reinterpret_cast<uintptr_t>(m->gate_out) | reinterpret_cast<uintptr_t>(m->kv);
  if (a16 & 15) return QSA_ERR_INVALID_ARG;
  p->main_qkv = static_cast<const uint16_t*>(m->qkv);
  p->main_q_norm_w = static_cast<const uint16_t*>(m->q_norm_w);
  p->main_k_norm_w = static_cast<const uint16_t*>(m->k_norm_w);
  p->main_eps = m->eps;
  p->main_q_out = static_cast<uint16_t*>(m->q_out);
  p->main_gate_out = static_cast<uint16_t*>(m->gate_out);
  p->main_kv = m->kv;
  p->main_slots = m->slot_mapping;
  p->main_hq = g->num_q_heads;
  p->main_hkv = g->num_kv_heads;
  p->main_page = g->page_size;
  p->main_blocks = g->num_blocks;
  p->main_kv_dtype = g->kv_dtype;
  p->main_k_scale = g->k_scale;
  p->main_v_scale = g->v_scale;
  return QSA_OK;
}

qsa_status do_compress(const qsa_cfg* cfg, const void* projected_q, void* q_idx,
                       const void* raw_keys, const int64_t* positions, const float* cos_sin,
                       const void* q_norm_w, const void* k_norm_w, void* ring, int32_t ring_blocks,
                       int64_t* ring_pos, const int32_t* ring_block_table, int32_t ring_bt_stride,
                       const int32_t* token_to_req, const int32_t* query_start_loc,
                       const int32_t* logical_positions, void* ccache, int32_t cpages,
                       const int64_t* compressed_slots, int32_t rows, int32_t reqs,
                       cudaStream_t stream, bool commit_ring = true,
                       CompressParams* out_params = nullptr,
                       const qsa_gqa_cfg* gcfg = nullptr, const qsa_main_prep* main = nullptr) {
  qsa_status st = check_cfg(cfg);
  if (st != QSA_OK) return st;
  if (rows < 0 || reqs < 0) return QSA_ERR_SHAPE;
  if (rows == 0) return QSA_OK;
  if (reqs < 1 || ring_blocks < 1 || cpages < 1 || ring_bt_stride < 1) return QSA_ERR_SHAPE;
  if ((projected_q == nullptr) != (q_idx == nullptr)) return QSA_ERR_INVALID_ARG;
  if (!raw_keys || !positions || !cos_sin || !q_norm_w || !k_norm_w || !ring ||
      !ring_block_table || !token_to_req || !query_start_loc || !logical_positions || !ccache ||
      !compressed_slots)
    return QSA_ERR_INVALID_ARG;
  const bool mrope = cfg->mrope_section[0] || cfg->mrope_section[1] || cfg->mrope_section[2];
  if (mrope != (ring_pos != nullptr)) return QSA_ERR_INVALID_ARG;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(raw_keys) | reinterpret_cast<uintptr_t>(ring) |
                        reinterpret_cast<uintptr_t>(ccache) | reinterpret_cast<uintptr_t>(q_norm_w) |
                        reinterpret_cast<uintptr_t>(k_norm_w) |
                        reinterpret_cast<uintptr_t>(projected_q) | reinterpret_cast<uintptr_t>(q_idx);
  if (a16 & 15) return QSA_ERR_INVALID_ARG;

  CompressParams p{};
  p.projected_q = static_cast<const uint16_t*>(projected_q);
  p.q_idx = q_idx;
  p.raw_keys = static_cast<const uint16_t*>(raw_keys);
  p.positions = positions;
  p.cos_sin = cos_sin;
  p.q_norm_w = static_cast<const uint16_t*>(q_norm_w);
  p.k_norm_w = static_cast<const uint16_t*>(k_norm_w);
  p.ring = static_cast<uint16_t*>(ring);
  p.ring_pos = ring_pos;
  p.ring_bt = ring_block_table;
  p.token_to_req = token_to_req;
  p.qsl = query_start_loc;
  p.logical = logical_positions;
  p.ccache = ccache;
  p.slots = compressed_slots;
  p.ring_blocks = ring_blocks;
  p.ring_bt_stride = ring_bt_stride;
  p.cpages = cpages;
  p.cpage = cfg->cpage;
  p.rows = rows;
  p.reqs = reqs;
  p.n_heads = cfg->n_heads;
  p.ratio = cfg->compress_ratio;
  p.S = cfg->state_size;
  p.max_pos = cfg->max_position;
  p.index_dtype = cfg->index_dtype;
  p.mrope = mrope ? 1 : 0;
  p.sec_h = cfg->mrope_section[1];
  p.sec_w = cfg->mrope_section[2];
  p.eps = cfg->eps;
  p.err = error_word();
  if (p.err == nullptr) return QSA_ERR_CUDA;
  if (main != nullptr) {
    st = fill_main(&p, gcfg, main);
    if (st != QSA_OK) return st;
  }
  if (out_params != nullptr) *out_params = p;
  if (t_validate_only) return QSA_OK;
  st = cuda_status(launch_compress(p, stream, /*pdl=*/false));
  if (st != QSA_OK || !commit_ring) return st;
  return cuda_status(launch_ring_commit(p, stream, /*pdl=*/true));
}

// Validates the logits arguments and fills the kernel parameters; the
// row-group table lives at the start of ws.
qsa_status logits_params(const qsa_cfg* cfg, const void* q_idx, const void* ccache, int32_t cpages,
                         const int32_t* cblock_table, int32_t cbt_stride,
                         const int32_t* token_to_req, const int32_t* query_start_loc,
                         const int32_t* logical_positions, float* logits, int64_t ld,
                         int32_t max_visible, int32_t rows, int32_t reqs, void* ws,
                         size_t ws_bytes, LogitsParams* out, int* npad_out, int* chunks_out,
                         int* groups_out) {
  qsa_status st = check_cfg(cfg);
  if (st != QSA_OK) return st;
  if (rows < 0 || reqs < 0 || max_visible < 0) return QSA_ERR_SHAPE;
  if (rows == 0 || max_visible == 0) return QSA_OK;
  if (reqs < 1 || cpages < 1 || cbt_stride < 1 || ld < max_visible) return QSA_ERR_SHAPE;
  if (!q_idx || !ccache || !cblock_table || !token_to_req || !query_start_loc ||
      !logical_positions || !logits)
    return QSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q_idx) | reinterpret_cast<uintptr_t>(ccache)) & 15)
    return QSA_ERR_INVALID_ARG;
  (void)ws;
  (void)ws_bytes;

  int R, npad;
  logits_grouping(cfg, rows, reqs, &R, &npad);
  // Two row groups per CTA share each key tile when the groups are full
  // (prefill-sized requests) and the e4m3 ring still fits beside two query
  // tiles.
  const int avg_rows = reqs > 0 ? (rows + reqs - 1) / reqs : 1;
  const int G = (cfg->index_dtype == QSA_DTYPE_E4M3 && npad == 256 && avg_rows >= 2 * R) ? 2 : 1;
  const int max_groups = max_groups_for(rows, reqs, R * G);
  LogitsParams p{};
  p.cblock_table = cblock_table;
  p.logical = logical_positions;
  p.qsl = query_start_loc;
  p.logits = logits;
  p.ccache = static_cast<const uint8_t*>(ccache);
  p.ld = ld;
  p.cbt_stride = cbt_stride;
  p.cpages = cpages;
  p.cpage = cfg->cpage;
  p.rows = rows;
  p.reqs = reqs;
  p.rows_per_group = R;
  p.groups_per_cta = G;
  p.n_heads = cfg->n_heads;
  p.ratio = cfg->compress_ratio;
  p.scale = 1.0f / (static_cast<float>(cfg->n_heads) * sqrtf(128.0f));
  p.row_bytes = 128 * elem_bytes(cfg);
  // One TMA box per compressed page needs pages of at least 8 keys (a box
  // then starts on a 1024-byte boundary of the swizzled tile) and row
  // coordinates within int32.
  p.tma_a = (cfg->cpage >= 8 && static_cast<long long>(cpages) * cfg->cpage < (1ll << 31)) ? 1 : 0;
  p.err = error_word();
  if (p.err == nullptr) return QSA_ERR_CUDA;
  p.token_to_req = token_to_req;
  p.remap = (R == 1 && G == 1 && npad <= 64) ? 1 : 0;

  const int max_tiles = (max_visible + 127) / 128;
  // Split each row group's key tiles into chunks so that the CTAs with work
  // (about ceil(rows / (R * G)) groups x chunks) fill one wave: 3 CTAs per SM
  // for the narrow kernels (N <= 64; 4 fit, but the compress kernel's CTAs
  // still hold registers on some SMs when they start: measured faster), 1 for
  // the wide ones (their shared memory and 256-512 TMEM columns).  The grid also holds the groups that a
  // ragged batch may need beyond that estimate; those CTAs leave at once.
  const long long slots = static_cast<long long>(sm_count()) * (npad <= 64 ? 3 : 1);
  const long long groups_est = (rows + static_cast<long long>(R) * G - 1) / (static_cast<long long>(R) * G);
  long long chunks_target = slots / (groups_est > 0 ? groups_est : 1);
  if (chunks_target < 1) chunks_target = 1;
  long long tpc = (max_tiles + chunks_target - 1) / chunks_target;
  if (tpc < 4) tpc = 4;  // amortise each CTA's set-up (measured on the long-context decode)
  if (tpc > max_tiles) tpc = max_tiles;
  if (tpc * (128 / cfg->cpage) > 4096) tpc = 4096 / (128 / cfg->cpage);
  p.tiles_per_cta = static_cast<int>(tpc);
  *chunks_out = static_cast<int>((max_tiles + tpc - 1) / tpc);
  *npad_out = npad;
  *groups_out = max_groups;
  *out = p;
  return QSA_OK;
}

qsa_status launch_logits(const qsa_cfg* cfg, const LogitsParams& p, const void* q_idx,
                         int32_t rows, int npad, int chunks, int max_groups, bool pdl,
                         cudaStream_t stream) {
  const int eb = elem_bytes(cfg);
  CUtensorMap tq, tcc;
  if (!encode_rows_map(&tq, q_idx, eb, static_cast<long long>(rows) * cfg->n_heads, npad))
    return QSA_ERR_CUDA;
  if (p.tma_a) {
    if (!encode_rows_map(&tcc, p.ccache, eb, static_cast<long long>(p.cpages) * p.cpage, p.cpage))
      return QSA_ERR_CUDA;
  } else {
    tcc = tq;  // unused
  }
  return cuda_status(launch_index_logits(p, tq, tcc, cfg->index_dtype, npad, max_groups, chunks,
                                         stream, pdl));
}

qsa_status do_logits(const qsa_cfg* cfg, const void* q_idx, const void* ccache, int32_t cpages,
                     const int32_t* cblock_table, int32_t cbt_stride, const int32_t* token_to_req,
                     const int32_t* query_start_loc, const int32_t* logical_positions,
                     float* logits, int64_t ld, int32_t max_visible, int32_t rows, int32_t reqs,
                     void* ws, size_t ws_bytes, cudaStream_t stream) {
  LogitsParams p{};
  int npad = 0, chunks = 0, groups = 0;
  qsa_status st = logits_params(cfg, q_idx, ccache, cpages, cblock_table, cbt_stride, token_to_req,
                                query_start_loc, logical_positions, logits, ld, max_visible, rows,
                                reqs, ws, ws_bytes, &p, &npad, &chunks, &groups);
  if (st != QSA_OK || rows == 0 || max_visible == 0) return st;
  return launch_logits(cfg, p, q_idx, rows, npad, chunks, groups, /*pdl=*/false, stream);
}

qsa_status do_topk(const qsa_cfg* cfg, const float* logits, int64_t ld, int32_t max_visible,
                   const int32_t* logical_positions, int32_t* packed, int32_t rows,
                   cudaStream_t stream, const CompressParams* ring = nullptr,
                   unsigned* tickets = nullptr, int tickets_per_row = 0, bool pdl = false) {
  qsa_status st = check_cfg(cfg);
  if (st != QSA_OK) return st;
  if (rows < 0 || max_visible < 0) return QSA_ERR_SHAPE;
  if (rows == 0) return QSA_OK;
  if (!logical_positions || !packed) return QSA_ERR_INVALID_ARG;
  const int kb = cfg->token_topk / cfg->compress_ratio;
  if (max_visible > kb && (!logits || ld < max_visible)) return QSA_ERR_INVALID_ARG;
  if (topk_smem_bytes(max_visible, kb) > topk_limit_bytes()) return QSA_ERR_UNSUPPORTED;
  TopkParams p{};
  p.logits = logits;
  p.ld = ld;
  p.logical = logical_positions;
  p.packed = packed;
  p.rows = rows;
  p.ratio = cfg->compress_ratio;
  p.token_topk = cfg->token_topk;
  p.max_visible = max_visible;
  p.err = error_word();
  if (p.err == nullptr) return QSA_ERR_CUDA;
  if (ring != nullptr) {
    p.do_ring = 1;
    p.ring = *ring;
  }
  p.tickets = tickets;
  p.tickets_per_row = tickets_per_row;
  p.sms = sm_count();
  if (t_validate_only) return QSA_OK;
  return cuda_status(launch_topk(p, stream, pdl));
}

qsa_status do_gqa(const qsa_gqa_cfg* gcfg, const void* q, const void* kv,
                  const int32_t* block_table, int32_t bt_stride, const int32_t* packed,
                  int32_t packed_width, const int32_t* token_to_req, const void* gate, void* out,
                  int32_t rows, void* ws, size_t ws_bytes, cudaStream_t stream,
                  bool pdl = false, bool tickets_zeroed = false, bool q_after_wait = false) {
  qsa_status st = check_gcfg(gcfg);
  if (st != QSA_OK) return st;
  if (rows < 0) return QSA_ERR_SHAPE;
  if (rows == 0) return QSA_OK;
  if (packed_width < 2 || bt_stride < 1) return QSA_ERR_SHAPE;
  if (!q || !kv || !block_table || !packed || !token_to_req || !out) return QSA_ERR_INVALID_ARG;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kv) |
                        reinterpret_cast<uintptr_t>(gate) | reinterpret_cast<uintptr_t>(out);
  if (a16 & 15) return QSA_ERR_INVALID_ARG;
  GqaParams p{};
  p.q = static_cast<const uint16_t*>(q);
  p.kv = kv;
  p.kv_dtype = gcfg->kv_dtype;
  p.k_scale = gcfg->k_scale;
  p.v_scale = gcfg->v_scale;
  p.q_after_wait = q_after_wait ? 1 : 0;
  p.block_table = block_table;
  p.packed = packed;
  p.token_to_req = token_to_req;
  p.gate = static_cast<const uint16_t*>(gate);
  p.out = static_cast<uint16_t*>(out);
  p.bt_stride = bt_stride;
  p.packed_width = packed_width;
  p.rows = rows;
  p.hq = gcfg->num_q_heads;
  p.hkv = gcfg->num_kv_heads;
  p.group = gcfg->num_q_heads / gcfg->num_kv_heads;
  p.page = gcfg->page_size;
  p.num_blocks = gcfg->num_blocks;
  const GqaLayout G = gqa_layout(gcfg, rows, packed_width);
  p.splits = G.splits;
  p.sms = sm_count();
  if (G.total > 0) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255)) return QSA_ERR_WORKSPACE;
    if (ws_bytes < G.total) return QSA_ERR_WORKSPACE;
    uint8_t* w = static_cast<uint8_t*>(ws);
    p.part_o = reinterpret_cast<float*>(w + G.po);
    p.part_lse = reinterpret_cast<float*>(w + G.pl);
    p.counters = reinterpret_cast<unsigned*>(w + G.tickets);
  }
  p.err = error_word();
  if (p.err == nullptr) return QSA_ERR_CUDA;
  if (t_validate_only) return QSA_OK;
  return cuda_status(launch_sparse_gqa(p, stream, pdl, !tickets_zeroed));
}

// Layer-step workspace regions.
struct StepLayout {
  size_t q_idx, logits, logits_ws, gqa_ws, total;
  long long ld;
};

bool step_layout(const qsa_cfg* c, const qsa_gqa_cfg* g, int rows, int reqs, int max_visible,
                 StepLayout* L) {
  if (check_cfg(c) != QSA_OK || check_gcfg(g) != QSA_OK) return false;
  if (rows < 0 || reqs < 0 || max_visible < 0) return false;
  const int pw = c->token_topk + c->compress_ratio;
  L->ld = logits_ld(max_visible);
  size_t off = 0;
  L->q_idx = off;
  off += align256(static_cast<size_t>(rows) * c->n_heads * 128 * elem_bytes(c));
  L->logits = off;
  off += align256(static_cast<size_t>(rows) * L->ld * sizeof(float));
  L->logits_ws = off;
  off += logits_ws_bytes(rows, reqs, c);
  L->gqa_ws = off;
  off += gqa_ws_bytes(g, rows, pw);
  L->total = off + 256;
  return true;
}

}  // namespace

// Error word of the current device, for entry points defined in other files.
unsigned long long* internal_error_word() { return error_word(); }

// Multiprocessors of the current device (queried once per device).
int sm_count() {
  static int count[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 152;
  if (count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    count[dev] = n;
  }
  return count[dev];
}


// Validation of the main-attention configuration, shared by every entry
// point that runs stage 4.
qsa_status check_gcfg(const qsa_gqa_cfg* g) {
  if (g == nullptr) return QSA_ERR_INVALID_ARG;
  if (g->head_dim != 128) return QSA_ERR_UNSUPPORTED;
  if (g->num_kv_heads < 1 || g->num_q_heads < g->num_kv_heads ||
      g->num_q_heads % g->num_kv_heads != 0)
    return QSA_ERR_SHAPE;
  const int group = g->num_q_heads / g->num_kv_heads;  // query heads per KV head
  if (group > 8 && group != 16) return QSA_ERR_UNSUPPORTED;
  if (g->page_size < 16 || g->page_size % 16 != 0) return QSA_ERR_SHAPE;
  if (g->num_blocks < 1) return QSA_ERR_SHAPE;
  if (g->kv_dtype != QSA_DTYPE_BF16 && g->kv_dtype != QSA_DTYPE_E4M3) return QSA_ERR_DTYPE;
  if (g->kv_dtype == QSA_DTYPE_E4M3 &&
      !(g->k_scale > 0.f && g->v_scale > 0.f && g->k_scale < 3.0e38f && g->v_scale < 3.0e38f))
    return QSA_ERR_INVALID_ARG;
  return QSA_OK;
}


}  // namespace qsa

using namespace qsa;

extern "C" {

qsa_status qsa_compress(const qsa_cfg* cfg, const void* projected_q, void* q_idx,
                        const void* raw_keys, const int64_t* positions, const float* cos_sin,
                        const void* q_norm_w, const void* k_norm_w, void* ring,
                        int32_t ring_blocks, int64_t* ring_pos,
                        const int32_t* ring_block_table, int32_t ring_bt_stride,
                        const int32_t* token_to_req, const int32_t* query_start_loc,
                        const int32_t* logical_positions, void* ccache, int32_t cpages,
                        const int64_t* compressed_slots, int32_t rows, int32_t reqs,
                        void* stream) {
  return do_compress(cfg, projected_q, q_idx, raw_keys, positions, cos_sin, q_norm_w, k_norm_w,
                     ring, ring_blocks, ring_pos, ring_block_table, ring_bt_stride, token_to_req,
                     query_start_loc, logical_positions, ccache, cpages, compressed_slots, rows,
                     reqs, static_cast<cudaStream_t>(stream));
}

qsa_status qsa_index_logits(const qsa_cfg* cfg, const void* q_idx, const void* ccache,
                            int32_t cpages, const int32_t* cblock_table, int32_t cbt_stride,
                            const int32_t* token_to_req, const int32_t* query_start_loc,
                            const int32_t* logical_positions, float* logits, int64_t ld,
                            int32_t max_visible, int32_t rows, int32_t reqs, void* ws,
                            size_t ws_bytes, void* stream) {
  return do_logits(cfg, q_idx, ccache, cpages, cblock_table, cbt_stride, token_to_req,
                   query_start_loc, logical_positions, logits, ld, max_visible, rows, reqs, ws,
                   ws_bytes, static_cast<cudaStream_t>(stream));
}

qsa_status qsa_topk(const qsa_cfg* cfg, const float* logits, int64_t ld, int32_t max_visible,
                    const int32_t* logical_positions, int32_t* packed, int32_t rows,
                    void* stream) {
  return do_topk(cfg, logits, ld, max_visible, logical_positions, packed, rows,
                 static_cast<cudaStream_t>(stream));
}

qsa_status qsa_sparse_gqa(const qsa_gqa_cfg* gcfg, const void* q, const void* kv,
                          const int32_t* block_table, int32_t bt_stride, const int32_t* packed,
                          int32_t packed_width, const int32_t* token_to_req, const void* gate,
                          void* out, int32_t rows, void* ws, size_t ws_bytes, void* stream) {
  return do_gqa(gcfg, q, kv, block_table, bt_stride, packed, packed_width, token_to_req, gate, out,
                rows, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

qsa_status qsa_layer_step(const qsa_cfg* cfg, const qsa_gqa_cfg* gcfg, const qsa_step_args* a,
                          int32_t skip_topk, void* ws, size_t ws_bytes, void* stream) {
  if (a == nullptr) return QSA_ERR_INVALID_ARG;
  qsa_status st = check_cfg(cfg);
  if (st != QSA_OK) return st;
  st = check_gcfg(gcfg);
  if (st != QSA_OK) return st;
  if (a->rows < 0 || a->reqs < 0) return QSA_ERR_SHAPE;
  if (a->packed == nullptr) return QSA_ERR_INVALID_ARG;
  if (a->rows == 0) return QSA_OK;
  StepLayout L;
  if (!step_layout(cfg, gcfg, a->rows, a->reqs, a->max_visible, &L)) return QSA_ERR_INVALID_ARG;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255)) return QSA_ERR_WORKSPACE;
  if (ws_bytes < L.total) return QSA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  const int pw = cfg->token_topk + cfg->compress_ratio;
  // stage 4's query and gate: the caller's, or the fused prepare's
  const qsa_main_prep* mp = a->main;
  if (mp != nullptr && mp->kv != a->kv) return QSA_ERR_INVALID_ARG;
  const void* q4 = mp != nullptr ? mp->q_out : a->q;
  const void* gate4 = mp != nullptr ? mp->gate_out : a->gate;
  const GqaLayout G = gqa_layout(gcfg, a->rows, pw);
  // Kernels after the first start early (programmatic dependent launch) and
  // wait on the device for their predecessor's results.
  if (skip_topk) {
    // stage 1 (ring commit included), then stage 4 on the given buffer
    st = do_compress(cfg, nullptr, nullptr, a->raw_keys, a->positions, a->cos_sin, a->q_norm_w,
                     a->k_norm_w, a->ring, a->ring_blocks, a->ring_pos, a->ring_block_table,
                     a->ring_bt_stride, a->token_to_req, a->query_start_loc, a->logical_positions,
                     a->ccache, a->cpages, a->compressed_slots, a->rows, a->reqs, s,
                     /*commit_ring=*/true, nullptr, gcfg, mp);
    if (st != QSA_OK) return st;
    return do_gqa(gcfg, q4, a->kv, a->block_table, a->bt_stride, a->packed, pw,
                  a->token_to_req, gate4, a->out, a->rows, w + L.gqa_ws, L.total - L.gqa_ws, s,
                  /*pdl=*/true, /*tickets_zeroed=*/false, /*q_after_wait=*/mp != nullptr);
  }
  void* q_idx = w + L.q_idx;
  float* logits = reinterpret_cast<float*>(w + L.logits);
  LogitsParams lp{};
  int npad = 0, chunks = 0, groups = 0;
  const bool any_visible = a->max_visible > 0;
  if (any_visible) {
    st = logits_params(cfg, q_idx, a->ccache, a->cpages, a->cblock_table, a->cbt_stride,
                       a->token_to_req, a->query_start_loc, a->logical_positions, logits, L.ld,
                       a->max_visible, a->rows, a->reqs, nullptr, 0, &lp, &npad, &chunks, &groups);
    if (st != QSA_OK) return st;
  }
  // stage 1 (the ring commit waits for the top-k launch)
  CompressParams cp{};
  st = do_compress(cfg, a->projected_q, q_idx, a->raw_keys, a->positions, a->cos_sin,
                   a->q_norm_w, a->k_norm_w, a->ring, a->ring_blocks, a->ring_pos,
                   a->ring_block_table, a->ring_bt_stride, a->token_to_req, a->query_start_loc,
                   a->logical_positions, a->ccache, a->cpages, a->compressed_slots, a->rows,
                   a->reqs, s, /*commit_ring=*/false, &cp, gcfg, mp);
  if (st != QSA_OK) return st;
  if (any_visible && !t_validate_only) {
    st = launch_logits(cfg, lp, q_idx, a->rows, npad, chunks, groups, /*pdl=*/true, s);
    if (st != QSA_OK) return st;
  }
  // stage 3; the same launch commits the ring after every pooling read and
  // clears the split-merge tickets of stage 4
  unsigned* tickets =
      G.total > 0 ? reinterpret_cast<unsigned*>(w + L.gqa_ws + G.tickets) : nullptr;
  st = do_topk(cfg, logits, L.ld, a->max_visible, a->logical_positions, a->packed, a->rows, s, &cp,
               tickets, tickets ? gcfg->num_kv_heads : 0, /*pdl=*/any_visible);
  if (st != QSA_OK) return st;
  return do_gqa(gcfg, q4, a->kv, a->block_table, a->bt_stride, a->packed, pw, a->token_to_req,
                gate4, a->out, a->rows, w + L.gqa_ws, L.total - L.gqa_ws, s, /*pdl=*/true,
                /*tickets_zeroed=*/tickets != nullptr, /*q_after_wait=*/mp != nullptr);
}

qsa_status qsa_qkv_index_proj(const void* x, const void* w, int32_t rows, int32_t hidden,
                              int32_t qkv_cols, int32_t index_q_cols, int32_t index_k_cols,
                              void* qkv_out, void* index_q_out, void* index_k_out, void* stream) {
  if (rows < 0 || hidden < 0 || qkv_cols < 0 || index_q_cols < 0 || index_k_cols < 0)
    return QSA_ERR_SHAPE;
  if (rows == 0) return QSA_OK;
  if (hidden < 64 || hidden % 64 != 0) return QSA_ERR_SHAPE;
  const long long ncols = static_cast<long long>(qkv_cols) + index_q_cols + index_k_cols;
  if (ncols < 1 || ncols >= (1ll << 31)) return QSA_ERR_SHAPE;
  if (!x || !w || (qkv_cols && !qkv_out) || (index_q_cols && !index_q_out) ||
      (index_k_cols && !index_k_out))
    return QSA_ERR_INVALID_ARG;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w);
  const uintptr_t a2 = reinterpret_cast<uintptr_t>(qkv_out) | reinterpret_cast<uintptr_t>(index_q_out) |
                       reinterpret_cast<uintptr_t>(index_k_out);
  if ((a16 & 15) || (a2 & 1)) return QSA_ERR_INVALID_ARG;
  ProjParams p{};
  p.qkv_out = static_cast<uint16_t*>(qkv_out);
  p.index_q_out = static_cast<uint16_t*>(index_q_out);
  p.index_k_out = static_cast<uint16_t*>(index_k_out);
  p.rows = rows;
  p.hidden = hidden;
  p.ncols = static_cast<int>(ncols);
  p.qkv_cols = qkv_cols;
  p.index_q_cols = index_q_cols;
  p.index_k_cols = index_k_cols;
  p.err = error_word();
  if (p.err == nullptr) return QSA_ERR_CUDA;
  CUtensorMap tw, tx;
  if (!encode_bf16_2d(&tw, w, hidden, ncols, 128) ||
      !encode_bf16_2d(&tx, x, hidden, rows, proj_x_box_rows(rows)))
    return QSA_ERR_CUDA;
  return cuda_status(launch_proj_gemm(p, tw, tx, static_cast<cudaStream_t>(stream)));
}

qsa_status qsa_main_prepare(const qsa_cfg* cfg, const qsa_gqa_cfg* gcfg, const qsa_main_prep* m,
                            const int64_t* positions, const float* cos_sin, int32_t rows,
                            void* stream) {
  qsa_status st = check_cfg(cfg);
  if (st != QSA_OK) return st;
  if (m == nullptr || rows < 0) return rows < 0 ? QSA_ERR_SHAPE : QSA_ERR_INVALID_ARG;
  if (rows == 0) return QSA_OK;
  if (!positions || !cos_sin) return QSA_ERR_INVALID_ARG;
  CompressParams p{};
  p.positions = positions;
  p.cos_sin = cos_sin;
  p.rows = rows;
  p.max_pos = cfg->max_position;
  p.mrope = (cfg->mrope_section[0] || cfg->mrope_section[1] || cfg->mrope_section[2]) ? 1 : 0;
  p.sec_h = cfg->mrope_section[1];
  p.sec_w = cfg->mrope_section[2];
  st = fill_main(&p, gcfg, m);
  if (st != QSA_OK) return st;
  p.err = error_word();
  if (p.err == nullptr) return QSA_ERR_CUDA;
  return cuda_status(launch_main_prepare(p, static_cast<cudaStream_t>(stream)));
}

qsa_status qsa_mtp_steps(const qsa_cfg* cfg, const qsa_gqa_cfg* gcfg, const qsa_step_args* steps,
                         int32_t k, void* ws, size_t ws_bytes, void* stream) {
  if (steps == nullptr || k < 1 || k > QSA_MTP_MAX_STEPS) return QSA_ERR_INVALID_ARG;
  for (int s = 1; s < k; ++s) {
    if (steps[s].rows != steps[0].rows || steps[s].reqs != steps[0].reqs ||
        steps[s].packed != steps[0].packed)
      return QSA_ERR_INVALID_ARG;
  }
  {
    ValidateOnly guard;  // every step is checked before the first launch
    for (int s = 0; s < k; ++s) {
      const qsa_status st = qsa_layer_step(cfg, gcfg, &steps[s], s > 0, ws, ws_bytes, stream);
      if (st != QSA_OK) return st;
    }
  }
  for (int s = 0; s < k; ++s) {
    const qsa_status st = qsa_layer_step(cfg, gcfg, &steps[s], s > 0, ws, ws_bytes, stream);
    if (st != QSA_OK) return st;
  }
  return QSA_OK;
}

size_t qsa_workspace_bytes(const qsa_cfg* cfg, const qsa_gqa_cfg* gcfg, int32_t rows,
                           int32_t reqs, int32_t max_visible) {
  StepLayout L;
  if (!step_layout(cfg, gcfg, rows, reqs, max_visible, &L)) return 0;
  return L.total;
}

int32_t qsa_step_launches(const qsa_cfg* cfg, const qsa_gqa_cfg* gcfg, int32_t rows,
                          int32_t reqs, int32_t skip_topk) {
  if (check_cfg(cfg) != QSA_OK || check_gcfg(gcfg) != QSA_OK || rows < 0 || reqs < 0) return 0;
  if (rows == 0) return 0;
  // split-KV partials are merged inside the GQA kernel
  return skip_topk ? 3 : 4;
}

int32_t qsa_gqa_splits(const qsa_gqa_cfg* gcfg, int32_t rows, int32_t packed_width) {
  if (check_gcfg(gcfg) != QSA_OK || rows <= 0 || packed_width < 2) return 0;
  return gqa_num_splits(rows, gcfg->num_kv_heads, packed_width, sm_count());
}

const char* qsa_status_string(qsa_status s) {
  switch (s) {
    case QSA_OK: return "ok";
    case QSA_ERR_INVALID_ARG: return "invalid argument (null pointer, misaligned or inconsistent)";
    case QSA_ERR_SHAPE: return "sizes do not fit together";
    case QSA_ERR_DTYPE: return "unsupported element type";
    case QSA_ERR_UNSUPPORTED: return "configuration not supported by this build";
    case QSA_ERR_WORKSPACE: return "workspace too small or not 256-byte aligned";
    case QSA_ERR_CUDA: return "CUDA runtime or launch error";
    case QSA_ERR_DEVICE_FAULT: return "device reported masked out-of-range accesses or a wait timeout";
  }
  return "unknown status";
}

qsa_status qsa_check_errors(int64_t* count) {
  if (count) *count = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return QSA_ERR_CUDA;
  unsigned long long* p = error_word();
  if (p == nullptr) return QSA_ERR_CUDA;
  unsigned long long v = 0, zero = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return QSA_ERR_CUDA;
  if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return QSA_ERR_CUDA;
  if (count) *count = static_cast<int64_t>(v);
  return v ? QSA_ERR_DEVICE_FAULT : QSA_OK;
}

const char* qsa_version(void) { return "qsa-gb300 0.1.0 (sm_103a)"; }

}  // extern "C"
