// Stage 3 of the QSA layer step: causal block top-k and expansion into the
// packed selection buffer.
//
// Follows "vllm.models.qwen4_exp.nvidia.qsa", QSAIndexer.forward (block
// indices of token_topk / compress_ratio columns over the row's visible
// blocks, then expand_qsa_block_indices) and the packed_output_width
// docstring: request-relative token indices padded with -1, trailing column
// = valid count.
//
// One CTA of 1024 threads per row.  The row's V logits are staged in shared
// memory as order-preserving 32-bit keys; an 8-bit radix select, starting
// below the bits that the row's smallest and largest keys share and with
// warp-aggregated histogram atomics, finds the K_b-th largest key T and how
// many keys equal to T are taken; a
// block-wide scan then writes the selected block ids in ascending order, the
// lower block winning among equal keys.  Rows with V <= K_b select every
// visible block without reading logits.
#include "qsa_device.cuh"
#include "qsa_kernels.h"
#include "stage_helpers.cuh"

namespace qsa {
namespace {

constexpr int kThreads = 1024;

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block scan of two counters at once.
__device__ __forceinline__ void block_scan2(int a, int b, int& ea, int& eb, int* wa, int* wb) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ia = a, ib = b;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int ya = __shfl_up_sync(0xffffffffu, ia, off);
    const int yb = __shfl_up_sync(0xffffffffu, ib, off);
    if (lane >= off) {
      ia += ya;
      ib += yb;
    }
  }
  if (lane == 31) {
    wa[warp] = ia;
    wb[warp] = ib;
  }
  __syncthreads();
  if (warp == 0) {
    int va = wa[lane], vb = wb[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int ya = __shfl_up_sync(0xffffffffu, va, off);
      const int yb = __shfl_up_sync(0xffffffffu, vb, off);
      if (lane >= off) {
        va += ya;
        vb += yb;
      }
    }
    wa[lane] = va;
    wb[lane] = vb;
  }
  __syncthreads();
  ea = (warp > 0 ? wa[warp - 1] : 0) + ia - a;
  eb = (warp > 0 ? wb[warp - 1] : 0) + ib - b;
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkParams P) {
  extern __shared__ uint32_t sm[];
  __shared__ int hist[256];
  __shared__ int s_digit, s_k;
  __shared__ int wa[32], wb[32];
  uint32_t* keys = sm;
  int* sel = reinterpret_cast<int*>(sm + P.max_visible);

  const int row = blockIdx.x, tid = threadIdx.x;
  const int r = P.ratio;
  const int kb = P.token_topk / r;
  const int W = P.token_topk + r - 1;
  int p = P.logical[row];
  if (p < -1) {
    if (tid == 0) flag_error(P.err);
    p = -1;
  }
  int V = (p + 1) / r;
  if (V > P.max_visible) {
    if (tid == 0) flag_error(P.err);
    V = P.max_visible;
    p = V * r - 1;
  }
  const bool take_all = V <= kb;
  if (!take_all) {
    const float* lrow = P.logits + static_cast<long long>(row) * P.ld;
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
    for (int c = tid; c < V; c += kThreads) {
      const uint32_t key = order_key(lrow[c]);
      keys[c] = key;
      kmin = min(kmin, key);
      kmax = max(kmax, key);
    }
    // Bits above the highest bit where the row's smallest and largest keys
    // differ are common to every key: the radix passes start below them.
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, off));
      kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, off));
    }
    if ((tid & 31) == 0) {
      wa[tid >> 5] = static_cast<int>(kmin);
      wb[tid >> 5] = static_cast<int>(kmax);
    }
    __syncthreads();
    if (tid < 32) {
      kmin = static_cast<uint32_t>(wa[tid]);
      kmax = static_cast<uint32_t>(wb[tid]);
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, off));
        kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, off));
      }
      if (tid == 0) {
        s_digit = static_cast<int>(kmin);
        s_k = static_cast<int>(kmax);
      }
    }
    __syncthreads();
    kmin = static_cast<uint32_t>(s_digit);
    kmax = static_cast<uint32_t>(s_k);
    __syncthreads();
    const uint32_t diff = kmin ^ kmax;
    int hi = diff ? 31 - __clz(diff) : -1;  // highest differing bit
    uint32_t prefix = hi >= 31 ? 0u : (kmin & ~((2u << hi) - 1u));
    uint32_t pmask = hi >= 31 ? 0u : ~((2u << hi) - 1u);
    if (hi < 0) {  // every key equal
      prefix = kmin;
      pmask = 0xFFFFFFFFu;
    }
    int k = kb;
    while (hi >= 0) {
      const int width = hi + 1 < 8 ? hi + 1 : 8;
      const int shift = hi - width + 1;
      const uint32_t dmask = (1u << width) - 1u;
      if (tid < 256) hist[tid] = 0;
      __syncthreads();
      for (int c = tid; c < V; c += kThreads) {
        const uint32_t key = keys[c];
        const bool in = (key & pmask) == prefix;
        const int bin = in ? static_cast<int>((key >> shift) & dmask) : -1;
        // lanes of a warp that fall in the same bin add once
        const unsigned active = __ballot_sync(__activemask(), in);
        if (in) {
          const unsigned same = __match_any_sync(active, bin);
          if ((threadIdx.x & 31) == __ffs(same) - 1) atomicAdd(&hist[bin], __popc(same));
        }
      }
      __syncthreads();
      if (tid < 32) {
        // lane l owns bins 255-8l .. 248-8l, scanned from the top
        int cnt[8], tot = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          cnt[j] = hist[255 - 8 * tid - j];
          tot += cnt[j];
        }
        int incl = tot;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, off);
          if (tid >= off) incl += y;
        }
        int cum = incl - tot;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (cum < k && k <= cum + cnt[j]) {
            s_digit = 255 - 8 * tid - j;
            s_k = k - cum;
          }
          cum += cnt[j];
        }
      }
      __syncthreads();
      prefix |= static_cast<uint32_t>(s_digit) << shift;
      pmask |= dmask << shift;
      k = s_k;
      hi = shift - 1;
      __syncthreads();
    }
    const uint32_t T = prefix;
    const int keq = k;

    const int per = (V + kThreads - 1) / kThreads;
    const int lo = min(V, tid * per), hi_end = min(V, lo + per);
    int gt = 0, eq = 0;
    for (int c = lo; c < hi_end; ++c) {
      const uint32_t key = keys[c];
      gt += key > T;
      eq += key == T;
    }
    int gt_ex, eq_ex;
    block_scan2(gt, eq, gt_ex, eq_ex, wa, wb);
    int out = gt_ex + min(eq_ex, keq);
    int eq_seen = eq_ex;
    for (int c = lo; c < hi_end; ++c) {
      const uint32_t key = keys[c];
      if (key > T) {
        sel[out++] = c;
      } else if (key == T) {
        if (eq_seen < keq) sel[out++] = c;
        ++eq_seen;
      }
    }
    __syncthreads();
  }

  const int nsel = take_all ? V : kb;
  const int tail0 = V * r;
  const int count = nsel * r + (p + 1 - tail0);
  int32_t* prow = P.packed + static_cast<long long>(row) * (W + 1);
  for (int idx = tid; idx < W; idx += kThreads) {
    int v = -1;
    if (idx < nsel * r) {
      const int b = take_all ? idx / r : sel[idx / r];
      v = b * r + idx % r;
    } else if (idx < count) {
      v = tail0 + (idx - nsel * r);
    }
    prow[idx] = v;
  }
  if (tid == 0) prow[W] = count;
  // Inside the layer step this launch also commits the row's raw key to the
  // compressor-state ring (all pooling reads of the step are done by now).
  if (P.do_ring && tid >= 32 && tid < 48) ring_commit_row(P.ring, row, tid - 32);
}

}  // namespace

size_t topk_smem_bytes(int max_visible, int block_topk) {
  return static_cast<size_t>(max_visible) * 4 + static_cast<size_t>(block_topk) * 4 + 16;
}

cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream) {
  if (p.rows == 0) return cudaSuccess;
  const size_t smem = topk_smem_bytes(p.max_visible, p.token_topk / p.ratio);
  cudaError_t e =
      cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  topk_kernel<<<p.rows, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace qsa
