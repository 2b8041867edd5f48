// Host-side launch interface between the C ABI (abi.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qsa.h"

namespace qsa {

// Defined in abi.cu, shared by the entry points of other files.
int sm_count();                                // multiprocessors of the current device
qsa_status check_gcfg(const qsa_gqa_cfg* g);   // main-attention configuration checks
unsigned long long* internal_error_word();     // device error word of the current device

struct CompressParams {
  const uint16_t* projected_q;  // [rows, n_heads*128] bf16 or null
  void* q_idx;                  // [rows, n_heads, 128] index dtype
  const uint16_t* raw_keys;     // [rows, 128] bf16
  const int64_t* positions;     // [rows, 3]
  const float* cos_sin;         // [max_pos, 64]
  const uint16_t* q_norm_w;     // [128]
  const uint16_t* k_norm_w;     // [128]
  uint16_t* ring;               // [ring_blocks, S, 128]
  int64_t* ring_pos;            // [ring_blocks, S, 3] or null
  const int32_t* ring_bt;       // [reqs, ring_bt_stride]
  const int32_t* token_to_req;
  const int32_t* qsl;
  const int32_t* logical;
  void* ccache;                 // [cpages, cpage, 128] index dtype
  const int64_t* slots;
  int ring_blocks, ring_bt_stride, cpages, cpage;
  int rows, reqs, n_heads, ratio, S, max_pos;
  int index_dtype, mrope, sec_h, sec_w;
  float eps;
  unsigned long long* err;
  // fused main-attention prepare (main_qkv == null: none)
  const uint16_t* main_qkv;     // [rows, (2 Hq + 2 Hkv) * 128] bf16
  const uint16_t* main_q_norm_w;
  const uint16_t* main_k_norm_w;
  float main_eps;
  uint16_t* main_q_out;         // [rows, Hq, 128] bf16
  uint16_t* main_gate_out;      // [rows, Hq, 128] bf16
  void* main_kv;                // [blocks, Hkv, page, 256] bf16 or e4m3
  const int64_t* main_slots;    // [rows] block * page + offset, < 0: no write
  int main_hq, main_hkv, main_page, main_blocks, main_kv_dtype;
  float main_k_scale, main_v_scale;
};

// pdl: launch with programmatic dependent launch (the kernel waits for the
// previous kernel on the stream before touching its results).
// With p.main_qkv set, the launch also prepares the main attention's q, gate
// and K/V cache rows (one more CTA per row).
cudaError_t launch_compress(const CompressParams& p, cudaStream_t stream, bool pdl);
// The main-attention prepare alone (one CTA per row).
cudaError_t launch_main_prepare(const CompressParams& p, cudaStream_t stream);
cudaError_t launch_ring_commit(const CompressParams& p, cudaStream_t stream, bool pdl);

struct LogitsParams {
  const int32_t* cblock_table;
  const int32_t* logical;
  const int32_t* qsl;
  float* logits;
  const uint8_t* ccache;  // compressed-key cache, gathered row by row
  long long ld;
  int cbt_stride, cpages, cpage;
  int rows, reqs, rows_per_group;
  int n_heads, ratio;
  float scale;
  int tiles_per_cta;
  int row_bytes;
  int tma_a;  // gather the key tiles with one TMA box per compressed page (cpage >= 8)
  int groups_per_cta;  // 1, or 2 (e4m3, N = 256): two row groups share each key tile
  // one row per group (decode): the CTAs, in launch order, take the (row, key
  // chunk) items that hold keys, so CTAs without work come last and leave
  int remap;
  const int32_t* token_to_req;  // [rows] request of each row (read when remap)
  unsigned long long* err;
};

// npad: padded MMA N (32, 64, 128 or 256); grid = (max_groups, chunks), CTA
// x handles row group x (each request's rows in chunks of rows_per_group *
// groups_per_cta).
// tmap_cc: the compressed cache as [cpages * cpage rows, 128 elements] with a
// box of cpage rows x 128 bytes (used when p.tma_a).
cudaError_t launch_index_logits(const LogitsParams& p, const CUtensorMap& tmap_q,
                                const CUtensorMap& tmap_cc, int index_dtype, int npad,
                                int max_groups, int chunks, cudaStream_t stream, bool pdl);

struct TopkParams {
  const float* logits;
  long long ld;
  const int32_t* logical;
  int32_t* packed;
  int rows, ratio, token_topk, max_visible;
  unsigned long long* err;
  int do_ring;            // also commit the step's raw keys to the ring
  CompressParams ring;
  unsigned* tickets;      // [rows, tickets_per_row] split-merge tickets to zero, or null
  int tickets_per_row;
  int sms;                // multiprocessors of the device (sizes the per-row clusters)
};
size_t topk_smem_bytes(int max_visible, int block_topk);
cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream, bool pdl);

struct GqaParams {
  const uint16_t* q;       // [rows, Hq, 128]
  const void* kv;          // [blocks, Hkv, page, 256] bf16 or e4m3 (kv_dtype)
  const int32_t* block_table;
  const int32_t* packed;
  const int32_t* token_to_req;
  const uint16_t* gate;    // nullable
  uint16_t* out;
  float* part_o;           // [splits, rows, Hq, 128]
  float* part_lse;         // [splits, rows, Hq]
  unsigned* counters;      // [rows, Hkv] merge tickets, or null for a separate merge launch
  int bt_stride, packed_width;
  int rows, hq, hkv, group, page, num_blocks, splits;  // group = hq / hkv: 1..8 or 16
  int kv_dtype;            // 0: bf16, 1: e4m3 with static scales
  float k_scale, v_scale;  // e4m3: stored value * scale = cached value
  int q_after_wait;        // q and gate are written by the kernels before this one
  int sms;                 // multiprocessors of the device (launch shape)
  unsigned long long* err;
};
// Split-KV factor for `rows` rows on a device with `sms` multiprocessors.
int gqa_num_splits(int rows, int hkv, int packed_width, int sms);
// zero_tickets: clear the merge tickets first (false when a preceding kernel
// of the same step already did).
cudaError_t launch_sparse_gqa(const GqaParams& p, cudaStream_t stream, bool pdl,
                              bool zero_tickets = true);

// The fused projection GEMM: y = x . w^T (bf16 in, fp32 accumulate, bf16
// out), output columns routed to the main qkv rows, then the indexer's query
// and key rows.
struct ProjParams {
  uint16_t* qkv_out;      // [rows, qkv_cols]
  uint16_t* index_q_out;  // [rows, index_q_cols]
  uint16_t* index_k_out;  // [rows, index_k_cols]
  int rows, hidden, ncols, qkv_cols, index_q_cols, index_k_cols;
  unsigned long long* err;
};
int proj_tile_rows(int rows);  // input rows per CTA tile (64, 128 or 256)
// input rows per TMA box: a tile's rows, or half of them for 256-row tiles
// (whose CTA pairs each load and multicast half)
int proj_x_box_rows(int rows);
// tmap_w: [ncols, hidden] bf16, box 64 x 128 rows; tmap_x: [rows, hidden]
// bf16, box 64 x proj_x_box_rows(rows) rows; both 128-byte swizzled.
cudaError_t launch_proj_gemm(const ProjParams& p, const CUtensorMap& tmap_w,
                             const CUtensorMap& tmap_x, cudaStream_t stream);

}  // namespace qsa
