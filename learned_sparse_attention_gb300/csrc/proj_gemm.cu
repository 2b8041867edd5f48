// The fused projection of the main attention and the indexer: one bf16 GEMM
// y = x . w^T over the stacked weights [w_qkv; w_index_q; w_index_k], the
// fp32 accumulator rounded once to bf16 and written to three outputs.
//
// Follows "vllm.models.qwen4_exp.nvidia.qsa": Qwen4ExpQSAQKVIndexerLinear
// (the indexer's index_qk_proj packed as shard 3 of the qkv GEMM, so one
// GEMM yields the sharded Q/gate, K and V and the replicated indexer Q/K),
// Qwen4ExpQSAAttention.forward (qkv, projected_qk = qkv.split([2 q_size +
// 2 kv_size, index_qk_size])) and QSAIndexer.forward (projected_q,
// raw_keys = projected_qk.split((index_n_heads D, index_kv_heads D))).
//
// GB300 mapping (tcgen05, swap-AB: the weights are the M = 128 operand, the
// input rows the N = 64 / 128 / 256 side, so a decode batch of 64 rows fills
// one N tile while 128 weight rows fill M).  One CTA per (128 output columns,
// BN input rows):
//   warp 0     one lane issues the TMA loads of each 64-element K slice of the
//              weight tile (128 rows x 128 B) and the input tile (BN rows x
//              128 B), 128-byte swizzled, into a ring of stages;
//   warp 1     allocates the TMEM accumulator (BN fp32 columns) and one lane
//              issues tcgen05.mma kind::f16 (four K = 16 steps per stage),
//              releasing each stage with tcgen05.commit;
//   warps 2-5  epilogue: each reads its 32 TMEM lanes (one output column
//              each) 32 input rows at a time, rounds to bf16 and stores; the
//              32 lanes of a warp write 32 consecutive columns of one row.
// Every wait is bounded (mbar_wait); a timeout sets the error word.
#include "qsa_device.cuh"
#include "qsa_kernels.h"
#include "qsa_launch.cuh"

namespace qsa {
namespace {

template <int BN>
struct ProjCfg {
  static constexpr int A_STAGE = 128 * 128;              // weight tile: 128 rows x 64 bf16
  static constexpr int B_STAGE = BN * 128;               // input tile: BN rows x 64 bf16
  static constexpr int STAGE = A_STAGE + B_STAGE;
  static constexpr int STAGES = (192 * 1024) / STAGE;    // 8 / 6 / 4
  static constexpr int THREADS = 192;
  static constexpr int SMEM = 1024 + STAGES * STAGE + 256;
  static_assert(STAGES >= 3, "ring depth");
};

// MC: the CTA pair of a 2-CTA cluster (adjacent 128-column tiles, the same
// BN input rows) shares the input tile: each CTA loads half of its rows and
// multicasts them to both, so a stage costs the SM's TMA unit A + B/2 bytes;
// a stage is free again once both CTAs' MMAs have read it (the commits are
// multicast onto both CTAs' empty barriers, which count two arrivals).
template <int BN, bool MC>
__global__ void __launch_bounds__(ProjCfg<BN>::THREADS, 1)
    proj_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w,
                     const __grid_constant__ CUtensorMap tmap_x, const ProjParams P) {
  using C = ProjCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
  uint8_t* sA = smem_raw + pad;
  uint8_t* sB = sA + C::STAGES * C::A_STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + C::STAGES * C::B_STAGE);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * 128;  // first output column (weight row)
  const int r0 = blockIdx.y * BN;   // first input row
  const int nk = P.hidden / 64;
  unsigned long long* err = P.err;

  const int crank = MC ? static_cast<int>(blockIdx.x & 1) : 0;  // rank in the CTA pair
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], MC ? 2 : 1);
    }
    mbar_init(acc_full, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, BN);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if constexpr (MC) cluster_sync_all();  // the peer's barriers exist before any multicast
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmap_w);
      tma_prefetch_desc(&tmap_x);
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % C::STAGES;
        const uint32_t ph = (kb / C::STAGES) & 1u;
        if (!mbar_wait(&empty[s], ph ^ 1u, err)) break;
        mbar_arrive_expect_tx(&full[s], C::STAGE);
        tma_load_2d(sA + s * C::A_STAGE, &tmap_w, kb * 64, n0, &full[s]);
        if constexpr (MC)  // this CTA's half of the input rows, to both CTAs
          tma_load_2d_multicast(sB + s * C::B_STAGE + crank * (C::B_STAGE / 2), &tmap_x, kb * 64,
                                r0 + crank * (BN / 2), &full[s], 0x3);
        else
          tma_load_2d(sB + s * C::B_STAGE, &tmap_x, kb * 64, r0, &full[s]);
      }
      if constexpr (MC) {
        // every stage released by both CTAs' MMAs before this CTA leaves: no
        // arrival from the peer may land on a barrier that no longer exists
        for (int kb = nk; kb < nk + C::STAGES; ++kb) {
          if (kb - C::STAGES < 0) continue;
          const int s = kb % C::STAGES;
          const uint32_t ph = (kb / C::STAGES) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, err)) break;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = umma_idesc(1u, 128, BN);  // bf16 x bf16 -> fp32
      const uint64_t a0 = umma_sdesc_sw128(smem_addr(sA));
      const uint64_t b0 = umma_sdesc_sw128(smem_addr(sB));
      bool ok = true;
      for (int kb = 0; kb < nk && ok; ++kb) {
        const int s = kb % C::STAGES;
        const uint32_t ph = (kb / C::STAGES) & 1u;
        ok = mbar_wait(&full[s], ph, err);
        if (!ok) break;
        tc_fence_after_sync();
        // the start-address field (address / 16, 14 bits) takes byte offsets
        // / 16 without carrying out (shared memory < 256 KB)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_f16(tmem, a0 + ((s * C::A_STAGE + kk * 32) >> 4), b0 + ((s * C::B_STAGE + kk * 32) >> 4),
                   idesc, (kb | kk) != 0 ? 1u : 0u);
        if constexpr (MC)
          umma_commit_multicast(&empty[s], 0x3);
        else
          umma_commit(&empty[s]);
      }
      umma_commit(acc_full);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int lane_base = 32 * (warp & 3);  // the TMEM lanes this warp may read
    const int col = n0 + lane_base + lane;   // this thread's output column
    const bool live = col < P.ncols;
    // output column -> (buffer, column, row stride)
    uint16_t* dst = nullptr;
    int dcol = 0, ld = 0;
    if (col < P.qkv_cols) {
      dst = P.qkv_out;
      dcol = col;
      ld = P.qkv_cols;
    } else if (col < P.qkv_cols + P.index_q_cols) {
      dst = P.index_q_out;
      dcol = col - P.qkv_cols;
      ld = P.index_q_cols;
    } else {
      dst = P.index_k_out;
      dcol = col - P.qkv_cols - P.index_q_cols;
      ld = P.index_k_cols;
    }
    if (mbar_wait(acc_full, 0, err)) {
      tc_fence_after_sync();
#pragma unroll 1
      for (int ch = 0; ch < BN / 32; ++ch) {
        uint32_t v[32];
        tmem_ld32_issue(tmem + (static_cast<uint32_t>(lane_base) << 16) + ch * 32, v);
        tmem_wait_ld32(v);
        const int rbase = r0 + ch * 32;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int row = rbase + j;
          if (live && row < P.rows) {
            const __nv_bfloat16 b = __float2bfloat16_rn(__uint_as_float(v[j]));
            dst[static_cast<long long>(row) * ld + dcol] = *reinterpret_cast<const uint16_t*>(&b);
          }
        }
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (MC) cluster_sync_all();  // the peer is done with this CTA's smem
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, BN);
  }
}

template <int BN, bool MC>
cudaError_t launch_bn(const ProjParams& p, const CUtensorMap& tw, const CUtensorMap& tx,
                      cudaStream_t stream) {
  using C = ProjCfg<BN>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(proj_gemm_kernel<BN, MC>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const int tiles_n = (p.ncols + 127) / 128;
  if constexpr (MC) {  // pairs of column tiles (an odd last one pairs with an empty tile)
    const dim3 grid((tiles_n + 1) / 2 * 2, (p.rows + BN - 1) / BN);
    return launch_kernel_cluster(proj_gemm_kernel<BN, MC>, grid, dim3(C::THREADS), C::SMEM, stream,
                                 false, 2, tw, tx, p);
  }
  const dim3 grid(tiles_n, (p.rows + BN - 1) / BN);
  return launch_kernel(proj_gemm_kernel<BN, MC>, grid, dim3(C::THREADS), C::SMEM, stream, false, tw,
                       tx, p);
}

}  // namespace

int proj_tile_rows(int rows) { return rows <= 64 ? 64 : rows <= 128 ? 128 : 256; }
int proj_x_box_rows(int rows) {
  const int t = proj_tile_rows(rows);
  return t == 256 ? t / 2 : t;
}

cudaError_t launch_proj_gemm(const ProjParams& p, const CUtensorMap& tmap_w,
                             const CUtensorMap& tmap_x, cudaStream_t stream) {
  if (p.rows == 0) return cudaSuccess;
  switch (proj_tile_rows(p.rows)) {
    case 64: return launch_bn<64, false>(p, tmap_w, tmap_x, stream);
    case 128: return launch_bn<128, false>(p, tmap_w, tmap_x, stream);
    default: return launch_bn<256, true>(p, tmap_w, tmap_x, stream);
  }
}

}  // namespace qsa
