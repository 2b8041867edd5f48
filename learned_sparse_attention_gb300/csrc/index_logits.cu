// Stage 2 of the QSA layer step: index logits on the tcgen05 tensor cores.
//
// Follows "vllm.models.qwen4_exp.nvidia.qsa", QSAIndexer.forward: the
// indexer query of each row is scored against the request's paged
// compressed-key cache (qsa_select_paged_decode / qsa_select_paged_prefill),
// weight-free: score(row, c) = (1 / (H * sqrt(D))) * sum_h relu(q_h . k_c),
// with fp8 x fp8 (plain e4m3, no scales) or bf16 x bf16 products.
//
// GB300 mapping.  The contraction is [keys x D] . [D x (rows*heads)], so the
// compressed keys are the M = 128 operand (A) and a group of rows of one
// request, all their heads, is the N operand (B), kept in shared memory for
// the whole CTA.  Per CTA:
//   warp 0      producer: TMA loads of the B tile once, then of 128-key A
//               tiles, one box per compressed page (pages are scattered, the
//               block table gives their physical index), into a 4-stage ring;
//   warp 1      allocates TMEM and issues tcgen05.mma (one thread), two
//               accumulator buffers so the epilogue overlaps the next tile;
//   warps 2..   epilogue: tcgen05.ld of the 128 x N accumulator, ReLU and
//               head-sum per row, scale, coalesced fp32 stores.
// Every wait is bounded (see mbar_wait); a timeout sets the error word.
#include "qsa_device.cuh"
#include "qsa_kernels.h"
#include "stage_helpers.cuh"

namespace qsa {
namespace {

template <int IDT, int NPAD>
struct LogitsCfg {
  static constexpr int ATOMS = IDT == 1 ? 1 : 2;        // 128-byte K atoms per key row
  static constexpr int A_ATOM = 128 * 128;              // bytes of one atom of a 128-key tile
  static constexpr int A_STAGE = A_ATOM * ATOMS;
  static constexpr int B_ATOM = NPAD * 128;
  static constexpr int B_BYTES = B_ATOM * ATOMS;
  static constexpr int STAGES = 4;
  static constexpr int EPI_WG = NPAD == 256 ? 2 : 1;
  static constexpr int THREADS = 64 + 128 * EPI_WG;
  static constexpr int KSTEPS = IDT == 1 ? 4 : 8;       // 32 bytes of K per MMA
  static constexpr uint32_t TMEM_COLS = 2 * NPAD;
  static constexpr int MAX_PAGES = 4096;                // page ids staged per CTA
  static constexpr int SMEM = 1024 + STAGES * A_STAGE + B_BYTES + 256 + MAX_PAGES * 4 + 32 * 4;
};

__global__ void __launch_bounds__(1024) logits_plan_kernel(const LogitsParams P) { plan_groups(P); }

template <int IDT, int NPAD>
__global__ void __launch_bounds__(LogitsCfg<IDT, NPAD>::THREADS, 1)
    index_logits_kernel(const __grid_constant__ CUtensorMap tmap_q,
                        const __grid_constant__ CUtensorMap tmap_k, const LogitsParams P) {
  using C = LogitsCfg<IDT, NPAD>;
  const int g = blockIdx.x;
  if (g >= *P.group_count) return;
  const int4 grp = P.groups[g];
  const int row0 = grp.x, nrows = grp.y, req = grp.z;
  const int p_last = P.logical[row0 + nrows - 1];
  const int vmax = p_last < 0 ? 0 : (p_last + 1) / P.ratio;
  const int total_tiles = (vmax + 127) / 128;
  const int t_begin = blockIdx.y * P.tiles_per_cta;
  const int t_end = min(total_tiles, t_begin + P.tiles_per_cta);
  if (t_begin >= t_end) return;
  const int ntiles = t_end - t_begin;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
  uint8_t* sA = smem_raw + pad;
  uint8_t* sB = sA + C::STAGES * C::A_STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + C::B_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* bar_q = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_q + 1);
  int* s_page = reinterpret_cast<int*>(smem_raw + pad + C::STAGES * C::A_STAGE + C::B_BYTES + 256);
  int* s_vis = s_page + C::MAX_PAGES;  // visible blocks of the group's rows

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cpage = P.cpage;
  const int32_t* bt_row = P.cblock_table + static_cast<long long>(req) * P.cbt_stride;
  // Prologue: the group's visible-block counts and the physical compressed
  // pages of this CTA's key range, resolved in parallel before any copy.
  const int ppt = P.manual ? 0 : 128 / cpage;  // pages per 128-key tile
  const int page0 = t_begin * ppt;
  const int npages = min(ntiles * ppt, C::MAX_PAGES);
  const int last_page = min((vmax - 1) / cpage, P.cbt_stride - 1);
  for (int i = threadIdx.x; i < npages; i += blockDim.x) {
    int phys = bt_row[min(page0 + i, last_page)];
    if (phys < 0 || phys >= P.cpages) {
      flag_error(P.err);
      phys = 0;
    }
    s_page[i] = phys;
  }
  for (int r = threadIdx.x; r < nrows; r += blockDim.x) {
    const int pr = P.logical[row0 + r];
    s_vis[r] = pr < 0 ? 0 : (pr + 1) / P.ratio;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 128 * C::EPI_WG);
    }
    mbar_init(bar_q, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  unsigned long long* err = P.err;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmap_q);
      tma_prefetch_desc(&tmap_k);
      mbar_arrive_expect_tx(bar_q, C::B_BYTES);
#pragma unroll
      for (int atom = 0; atom < C::ATOMS; ++atom)
        tma_load_2d(sB + atom * C::B_ATOM, &tmap_q, atom * 64, row0 * P.n_heads, bar_q);
    }
    for (int i = 0; i < ntiles; ++i) {
      const int s = i % C::STAGES;
      const uint32_t ph = (i / C::STAGES) & 1;
      if (!mbar_wait(&empty[s], ph ^ 1, err)) break;
      const int tile = t_begin + i;
      uint8_t* dst = sA + s * C::A_STAGE;
      if (!P.manual) {
        const int pages = 128 / cpage;
        if (lane == 0) mbar_arrive_expect_tx(&full[s], C::A_STAGE);
        __syncwarp();
        for (int pg = lane; pg < pages; pg += 32) {
          const int phys = s_page[min(i * pages + pg, npages - 1)];
#pragma unroll
          for (int atom = 0; atom < C::ATOMS; ++atom)
            tma_load_2d(dst + atom * C::A_ATOM + pg * cpage * 128, &tmap_k, atom * 64,
                        phys * cpage, &full[s]);
        }
      } else {
        // Copy path for pages shorter than one 8-row swizzle group: plain
        // 16-byte loads written in the same 128-byte swizzled layout.
        constexpr int CHUNKS = 8 * C::ATOMS;
        for (int idx = lane; idx < 128 * CHUNKS; idx += 32) {
          const int m = idx / CHUNKS, c = idx % CHUNKS;
          const int atom = c >> 3, cc = c & 7;
          const int key = tile * 128 + m;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (key < vmax && key / cpage < P.cbt_stride) {
            const int phys = bt_row[key / cpage];
            if (phys >= 0 && phys < P.cpages) {
              const uint8_t* src = P.ccache +
                                   (static_cast<long long>(phys) * cpage + key % cpage) * P.row_bytes +
                                   c * 16;
              v = *reinterpret_cast<const uint4*>(src);
            } else if (cc == 0 && atom == 0) {
              flag_error(err);
            }
          }
          *reinterpret_cast<uint4*>(dst + atom * C::A_ATOM + m * 128 + ((cc ^ (m & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t n_eff = ((nrows * P.n_heads + 31) / 32) * 32;
      if (n_eff > NPAD) n_eff = NPAD;
      const uint32_t idesc = umma_idesc(IDT == 1 ? 0u : 1u, 128, n_eff);
      bool ok = mbar_wait(bar_q, 0, err);
      const uint32_t b_base = smem_addr(sB);
      for (int i = 0; ok && i < ntiles; ++i) {
        const int s = i % C::STAGES;
        const uint32_t ph = (i / C::STAGES) & 1;
        const int a = i & 1;
        const uint32_t aph = (i >> 1) & 1;
        if (!mbar_wait(&acc_empty[a], aph ^ 1, err)) break;
        if (!mbar_wait(&full[s], ph, err)) break;
        tc_fence_after_sync();
        const uint32_t a_base = smem_addr(sA + s * C::A_STAGE);
        const uint32_t d_tmem = tmem_base + a * NPAD;
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {
          const uint32_t atom = kk >> 2, koff = (kk & 3) * 32;
          const uint64_t adesc = umma_sdesc_sw128(a_base + atom * C::A_ATOM + koff);
          const uint64_t bdesc = umma_sdesc_sw128(b_base + atom * C::B_ATOM + koff);
          if (IDT == 1)
            umma_f8f6f4(d_tmem, adesc, bdesc, idesc, kk > 0 ? 1u : 0u);
          else
            umma_f16(d_tmem, adesc, bdesc, idesc, kk > 0 ? 1u : 0u);
        }
        umma_commit(&empty[s]);
        umma_commit(&acc_full[a]);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int wg = (warp - 2) >> 2;
    const int lane_base = 32 * (warp & 3);
    const int m = lane_base + lane;
    const int cols = nrows * P.n_heads;
    const int col_begin = wg * (NPAD / C::EPI_WG);
    const int col_end = min(cols, col_begin + NPAD / C::EPI_WG);
    constexpr int COLS = NPAD / C::EPI_WG;  // accumulator columns of this warpgroup
    for (int i = 0; i < ntiles; ++i) {
      const int a = i & 1;
      const uint32_t aph = (i >> 1) & 1;
      if (!mbar_wait(&acc_full[a], aph, err)) break;
      tc_fence_after_sync();
      const int key = (t_begin + i) * 128 + m;
      // One wide TMEM read of the warpgroup's columns, then the accumulator
      // goes straight back to the MMA warp; sums and stores follow.
      float v[COLS];
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(lane_base) << 16) + a * NPAD + col_begin;
      if constexpr (COLS == 32) tmem_ld32(taddr, v);
      else if constexpr (COLS == 64) tmem_ld64_wait(taddr, v);
      else tmem_ld128_wait(taddr, v);
      tc_fence_before_sync();
      mbar_arrive_relaxed(&acc_empty[a]);
      // ReLU sums of 8-column segments, then a pairwise tree up to n_heads
      // columns per row (n_heads is 8, 16, 32 or 64): branch-free, compact.
      constexpr int NSEG = COLS / 8;
      float seg[NSEG];
#pragma unroll
      for (int q = 0; q < NSEG; ++q) {
        float t = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) t += fmaxf(v[q * 8 + e], 0.f);
        seg[q] = t;
      }
      if (P.n_heads >= 16) {
#pragma unroll
        for (int q = 0; q < NSEG / 2; ++q) seg[q] = seg[2 * q] + seg[2 * q + 1];
      }
      if (P.n_heads >= 32) {
#pragma unroll
        for (int q = 0; q < NSEG / 4; ++q) seg[q] = seg[2 * q] + seg[2 * q + 1];
      }
      if (P.n_heads >= 64) {
#pragma unroll
        for (int q = 0; q < NSEG / 8; ++q) seg[q] = seg[2 * q] + seg[2 * q + 1];
      }
      const int rows_here = max(0, col_end - col_begin) / P.n_heads;
      const int r0 = col_begin / P.n_heads;
#pragma unroll
      for (int q = 0; q < NSEG; ++q) {
        if (q < rows_here) {
          const int r = r0 + q;
          if (r < nrows && key < s_vis[r])
            P.logits[static_cast<long long>(row0 + r) * P.ld + key] = seg[q] * P.scale;
        }
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <int IDT, int NPAD>
cudaError_t launch_one(const LogitsParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                       int max_groups, int chunks, cudaStream_t stream) {
  using C = LogitsCfg<IDT, NPAD>;
  auto kern = index_logits_kernel<IDT, NPAD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<dim3(max_groups, chunks), C::THREADS, C::SMEM, stream>>>(tq, tk, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_logits_plan(const LogitsParams& p, cudaStream_t stream) {
  logits_plan_kernel<<<1, 1024, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_index_logits(const LogitsParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                                int index_dtype, int npad, int max_groups, int chunks,
                                cudaStream_t stream) {
  if (max_groups <= 0 || chunks <= 0) return cudaSuccess;
  if (index_dtype == 1) {
    switch (npad) {
      case 32: return launch_one<1, 32>(p, tq, tk, max_groups, chunks, stream);
      case 64: return launch_one<1, 64>(p, tq, tk, max_groups, chunks, stream);
      case 128: return launch_one<1, 128>(p, tq, tk, max_groups, chunks, stream);
      case 256: return launch_one<1, 256>(p, tq, tk, max_groups, chunks, stream);
    }
  } else {
    switch (npad) {
      case 32: return launch_one<0, 32>(p, tq, tk, max_groups, chunks, stream);
      case 64: return launch_one<0, 64>(p, tq, tk, max_groups, chunks, stream);
      case 128: return launch_one<0, 128>(p, tq, tk, max_groups, chunks, stream);
      case 256: return launch_one<0, 256>(p, tq, tk, max_groups, chunks, stream);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace qsa
