// Stage 1 of the QSA layer step: indexer query prep, group pooling into the
// compressed-key cache and the compressor-state ring commit.
//
// Follows "vllm.models.qwen4_exp.nvidia.qsa", QSAIndexer.forward (unfused
// reference path: gemma_rmsnorm -> apply_qsa_rope -> cast for the query;
// qsa_compress_groups_with_ratio -> gemma_rmsnorm -> RoPE at the group's first
// position -> cast -> qsa_store_cache_rows for the compressed key, the raw key
// and the rope position) and "indexer_qsa.py", apply_qsa_rope (NeoX pairs
// (i, i + rotary_dim/2), cos|sin halves of the caller's table, interleaved
// MRoPE).  The norm, rotation and cast are fused into one pass in fp32 with a
// single rounding to the indexer dtype.
//
// Layout of the work: 128-thread CTAs.  CTA i < rows prepares the query of
// row i: 8 half-warps, each owning n_heads / 8 head vectors, each lane 8
// consecutive dims (one 16-byte load per head, all issued before any math);
// RoPE partners (i, i + 32) sit 4 lanes apart.  CTA rows + i pools the group
// completed by row i, if any, in parallel with the query CTAs.  With the fused
// main-attention prepare, CTA 2 rows + i prepares row i's main q, gate and
// K/V cache rows (caller inputs only, so it does not wait for anything).
#include "qsa_device.cuh"
#include "qsa_kernels.h"
#include "qsa_launch.cuh"
#include "stage_helpers.cuh"
#include "qsa_rope.cuh"

namespace qsa {
namespace {

constexpr int kD = 128;

template <int IDT>
__device__ __forceinline__ void store8(void* base, long long elem_off, const float (&x)[8]) {
  if (IDT == 1) {
    uint2 v;
    v.x = static_cast<uint32_t>(f32x2_to_e4m3x2(x[0], x[1])) |
          (static_cast<uint32_t>(f32x2_to_e4m3x2(x[2], x[3])) << 16);
    v.y = static_cast<uint32_t>(f32x2_to_e4m3x2(x[4], x[5])) |
          (static_cast<uint32_t>(f32x2_to_e4m3x2(x[6], x[7])) << 16);
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(base) + elem_off) = v;
  } else {
    uint4 v;
    v.x = pack_bf16x2(x[0], x[1]);
    v.y = pack_bf16x2(x[2], x[3]);
    v.z = pack_bf16x2(x[4], x[5]);
    v.w = pack_bf16x2(x[6], x[7]);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + elem_off) = v;
  }
}

// Main-attention prepare of one row by a 128-thread CTA (8 half-warps, each
// a 128-dim head vector, 8 dims per lane): q = RoPE(GemmaRMSNorm(q)) -> bf16,
// the gate passed through, k = RoPE(GemmaRMSNorm(k)) and v written into the
// paged KV cache at the row's slot (bf16, or e4m3(x / scale)).  Follows
// "vllm.models.qwen4_exp.nvidia.qsa", QSAIndexer.forward (the qsa_prepare
// call: main_qkv, main_q_norm_weight, main_k_norm_weight, main_eps,
// main_kv_cache, main_slot_mapping, main_k_scale, main_v_scale) and
// Qwen4ExpQSAAttention.__init__ (the gate packed next to each query head,
// q_norm / k_norm per head, the indexer's rotary embedding).
__device__ __forceinline__ void main_prepare_row(const CompressParams& P, int row) {
  const int hw = threadIdx.x >> 4, lane16 = threadIdx.x & 15;
  const int HQ = P.main_hq, HKV = P.main_hkv;
  const uint16_t* x = P.main_qkv + static_cast<long long>(row) * (2 * HQ + 2 * HKV) * kD;
  int64_t pos[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) pos[k] = P.positions[static_cast<long long>(row) * 3 + (P.mrope ? k : 0)];
  float c[8], s[8], wq[8], wk[8];
  rope_coeffs(rope_params(P), lane16, pos, c, s);
  load8_bf16(P.main_q_norm_w + 8 * lane16, wq);
  load8_bf16(P.main_k_norm_w + 8 * lane16, wk);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    wq[e] += 1.0f;
    wk[e] += 1.0f;
  }
  // query heads (both half-warps of a warp run the same iterations: the
  // norm's shuffles span the warp)
  for (int base = 0; base < HQ; base += 8) {
    const int h = base + hw;
    const bool act = h < HQ;
    float xq[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    uint4 gv = make_uint4(0u, 0u, 0u, 0u);
    if (act) {
      load8_bf16(x + (2 * h) * kD + 8 * lane16, xq);
      gv = *reinterpret_cast<const uint4*>(x + (2 * h + 1) * kD + 8 * lane16);
    }
    norm_rope(xq, wq, P.main_eps, lane16, c, s);
    if (act) {
      const long long o = (static_cast<long long>(row) * HQ + h) * kD + 8 * lane16;
      store8<0>(P.main_q_out, o, xq);
      *reinterpret_cast<uint4*>(P.main_gate_out + o) = gv;
    }
  }
  // K and V into the cache at the row's slot
  const long long slot = P.main_slots[row];
  if (slot < 0) return;
  const long long blk = slot / P.main_page, off = slot - blk * P.main_page;
  if (blk >= P.main_blocks) {
    if (threadIdx.x == 0) flag_error(P.err);
    return;
  }
  for (int base = 0; base < HKV; base += 8) {
    const int h = base + hw;
    const bool act = h < HKV;
    float xk[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    uint4 vv = make_uint4(0u, 0u, 0u, 0u);
    if (act) {
      load8_bf16(x + (2 * HQ + h) * kD + 8 * lane16, xk);
      vv = *reinterpret_cast<const uint4*>(x + (2 * HQ + HKV + h) * kD + 8 * lane16);
    }
    norm_rope(xk, wk, P.main_eps, lane16, c, s);
    if (!act) continue;
    const long long r = (blk * HKV + h) * P.main_page + off;  // (token, KV head) row
    if (P.main_kv_dtype == 0) {
      uint16_t* dst = static_cast<uint16_t*>(P.main_kv) + r * 256;
      store8<0>(dst, 8 * lane16, xk);
      *reinterpret_cast<uint4*>(dst + 128 + 8 * lane16) = vv;
    } else {
      uint8_t* dst = static_cast<uint8_t*>(P.main_kv) + r * 256;
      const float ik = 1.0f / P.main_k_scale, iv = 1.0f / P.main_v_scale;
      float xv[8] = {bf16_lo(vv.x), bf16_hi(vv.x), bf16_lo(vv.y), bf16_hi(vv.y),
                     bf16_lo(vv.z), bf16_hi(vv.z), bf16_lo(vv.w), bf16_hi(vv.w)};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        xk[e] *= ik;
        xv[e] *= iv;
      }
      store8<1>(dst, 8 * lane16, xk);
      store8<1>(dst, 128 + 8 * lane16, xv);
    }
  }
}

// IDT: indexer dtype (0 bf16, 1 e4m3); NHH: query heads per half-warp
// (n_heads / 8), so that the query's registers fit the head count: fewer
// registers, more CTAs per SM for long prefill chunks.
template <int IDT, int NHH>
__global__ void __launch_bounds__(128) compress_kernel(const CompressParams P) {
  griddep_launch_dependents();
  if (blockIdx.x >= 2 * P.rows) {  // reads only caller inputs: no wait
    main_prepare_row(P, blockIdx.x - 2 * P.rows);
    return;
  }
  griddep_wait();
  const int b = blockIdx.x;
  const bool pool = b >= P.rows;
  const int row = pool ? b - P.rows : b;
  const int hw = threadIdx.x >> 4;       // half-warp 0..7
  const int lane16 = threadIdx.x & 15;   // dims 8*lane16 .. +7
  // the row's metadata in one round trip (the pooling CTAs' slot with it)
  const int req = P.token_to_req[row];
  const int p = P.logical[row];
  const long long slot = pool ? P.slots[row] : -1;

  if (!pool) {
    // ---- indexer query: every head of this row, all loads issued first
    // (they read only this row's caller inputs, so they go out before the
    // request id is checked)
    if (P.projected_q == nullptr) return;
    float x[NHH][8];
#pragma unroll
    for (int k = 0; k < NHH; ++k)
      load8_bf16(P.projected_q + (static_cast<long long>(row) * P.n_heads + hw + 8 * k) * kD +
                     8 * lane16, x[k]);
    int64_t pos[3];
#pragma unroll
    for (int k = 0; k < 3; ++k)
      pos[k] = P.positions[static_cast<long long>(row) * 3 + (P.mrope ? k : 0)];
    float c[8], s[8], w1[8];
    load8_bf16(P.q_norm_w + 8 * lane16, w1);
    if (req < 0 || req >= P.reqs) return;
    rope_coeffs(rope_params(P), lane16, pos, c, s);
#pragma unroll
    for (int e = 0; e < 8; ++e) w1[e] += 1.0f;
#pragma unroll
    for (int k = 0; k < NHH; ++k) {
      norm_rope(x[k], w1, P.eps, lane16, c, s);
      store8<IDT>(P.q_idx,
                  (static_cast<long long>(row) * P.n_heads + hw + 8 * k) * kD + 8 * lane16, x[k]);
    }
    return;
  }

  // ---- group completed by this row: pool, norm, rotate, cast, store.
  // Warp 0 runs it; both of its half-warps compute the same key (the
  // shuffles stay inside a half-warp) and half-warp 0 stores it.
  if (req < 0 || req >= P.reqs) {
    if (threadIdx.x == 0) flag_error(P.err);
    return;
  }
  if (slot < 0 || (threadIdx.x >> 5) != 0) return;
  const int r = P.ratio;
  const int first_row = P.qsl[req];
  const int ring_block = P.ring_bt[static_cast<long long>(req) * P.ring_bt_stride];
  if (first_row < 0 || first_row > row) {  // inconsistent query_start_loc
    if (threadIdx.x == 0) flag_error(P.err);
    return;
  }
  const int step_start = P.logical[first_row];
  const long long nslots = static_cast<long long>(P.cpages) * P.cpage;
  const int t0 = p - r + 1;
  const bool ring_needed = t0 < step_start;
  // raw keys of this step are rows first_row .. first_row + (p - step_start),
  // which must not pass this row
  if (slot >= nslots || t0 < 0 || p - step_start > row - first_row ||
      (ring_needed && (ring_block < 0 || ring_block >= P.ring_blocks))) {
    if (threadIdx.x == 0) flag_error(P.err);
    return;
  }
  // The group's keys go out 8 at a time (one round trip for r <= 8) and
  // are summed in position order, together with the RoPE position's loads.
  uint4 kr[8];
  auto load_keys = [&](int tb) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int t = tb + u;
      if (t > p) continue;
      const uint16_t* src =
          t >= step_start ? P.raw_keys + static_cast<long long>(first_row + (t - step_start)) * kD
                          : P.ring + (static_cast<long long>(ring_block) * P.S + (t % P.S)) * kD;
      kr[u] = *reinterpret_cast<const uint4*>(src + 8 * lane16);
    }
  };
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  auto sum_keys = [&](int tb) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (tb + u > p) continue;
      acc[0] += bf16_lo(kr[u].x); acc[1] += bf16_hi(kr[u].x);
      acc[2] += bf16_lo(kr[u].y); acc[3] += bf16_hi(kr[u].y);
      acc[4] += bf16_lo(kr[u].z); acc[5] += bf16_hi(kr[u].z);
      acc[6] += bf16_lo(kr[u].w); acc[7] += bf16_hi(kr[u].w);
    }
  };
  load_keys(t0);

  int64_t pos[3];
  if (!P.mrope) {
    pos[0] = pos[1] = pos[2] = t0;
  } else if (t0 >= step_start) {
    const long long src_row = first_row + (t0 - step_start);
#pragma unroll
    for (int k = 0; k < 3; ++k) pos[k] = P.positions[src_row * 3 + k];
  } else {
    const long long ring_slot = static_cast<long long>(ring_block) * P.S + (t0 % P.S);
#pragma unroll
    for (int k = 0; k < 3; ++k) pos[k] = P.ring_pos[ring_slot * 3 + k];
  }
  float c[8], s[8], w1[8];
  load8_bf16(P.k_norm_w + 8 * lane16, w1);
  rope_coeffs(rope_params(P), lane16, pos, c, s);
  sum_keys(t0);
  for (int tb = t0 + 8; tb <= p; tb += 8) {
    load_keys(tb);
    sum_keys(tb);
  }
  const float inv_r = 1.0f / static_cast<float>(r);
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] *= inv_r;
#pragma unroll
  for (int e = 0; e < 8; ++e) w1[e] += 1.0f;
  norm_rope(acc, w1, P.eps, lane16, c, s);
  if (hw == 0) store8<IDT>(P.ccache, slot * kD + 8 * lane16, acc);
}

// Ring commit: runs after every pooling read of the step.  Each request's
// newest S raw keys (and 3-D positions) go to their ring slots.  A row writes
// only if no later row of its request maps to the same slot, which gives the
// sequential "later rows overwrite earlier rows" result without races.
__global__ void __launch_bounds__(128) ring_commit_kernel(const CompressParams P) {
  griddep_launch_dependents();
  griddep_wait();  // every pooling read of the compress kernel is done
  const int row = blockIdx.x * 8 + (threadIdx.x >> 4);
  if (row < P.rows) ring_commit_row(P, row, threadIdx.x & 15);
}

__global__ void __launch_bounds__(128) main_prepare_kernel(const CompressParams P) {
  main_prepare_row(P, blockIdx.x);
}

}  // namespace

template <int IDT>
cudaError_t launch_compress_dt(const CompressParams& p, dim3 grid, cudaStream_t stream, bool pdl) {
  switch (p.n_heads >> 3) {
    case 1: return launch_kernel(compress_kernel<IDT, 1>, grid, dim3(128), 0, stream, pdl, p);
    case 2: return launch_kernel(compress_kernel<IDT, 2>, grid, dim3(128), 0, stream, pdl, p);
    case 4: return launch_kernel(compress_kernel<IDT, 4>, grid, dim3(128), 0, stream, pdl, p);
    case 8: return launch_kernel(compress_kernel<IDT, 8>, grid, dim3(128), 0, stream, pdl, p);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_compress(const CompressParams& p, cudaStream_t stream, bool pdl) {
  if (p.rows == 0) return cudaSuccess;
  const dim3 grid((p.main_qkv != nullptr ? 3 : 2) * p.rows);
  if (p.index_dtype == 1) return launch_compress_dt<1>(p, grid, stream, pdl);
  return launch_compress_dt<0>(p, grid, stream, pdl);
}

cudaError_t launch_main_prepare(const CompressParams& p, cudaStream_t stream) {
  if (p.rows == 0) return cudaSuccess;
  return launch_kernel(main_prepare_kernel, dim3(p.rows), dim3(128), 0, stream, false, p);
}

cudaError_t launch_ring_commit(const CompressParams& p, cudaStream_t stream, bool pdl) {
  if (p.rows == 0) return cudaSuccess;
  return launch_kernel(ring_commit_kernel, dim3((p.rows + 7) / 8), dim3(128), 0, stream, pdl, p);
}

}  // namespace qsa
