// Stage 3 of the QSA layer step: causal block top-k and expansion into the
// packed selection buffer.
//
// Follows "vllm.models.qwen4_exp.nvidia.qsa", QSAIndexer.forward (block
// indices of token_topk / compress_ratio columns over the row's visible
// blocks, then expand_qsa_block_indices) and the packed_output_width
// docstring: request-relative token indices padded with -1, trailing column
// = valid count.
//
// Shared-memory variant (rows longer than the register variant covers): one
// CTA of 1024 threads per row.  The row's V logits are staged in shared
// memory as order-preserving 32-bit keys; an 8-bit radix select, starting
// below the bits that the row's smallest and largest keys share and with
// warp-aggregated histogram atomics, finds the K_b-th largest key T and how
// many keys equal to T are taken; a
// block-wide scan then writes the selected block ids in ascending order, the
// lower block winning among equal keys.  Rows with V <= K_b select every
// visible block without reading logits.
#include <cooperative_groups.h>

#include "qsa_device.cuh"
#include "qsa_kernels.h"
#include "qsa_launch.cuh"
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

  griddep_launch_dependents();
  if (P.tickets != nullptr && threadIdx.x < P.tickets_per_row)
    P.tickets[static_cast<long long>(blockIdx.x) * P.tickets_per_row + threadIdx.x] = 0u;
  griddep_wait();  // logits (and, transitively, the compress kernel) are done
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


// ---------------------------------------------------------------------------
// Register variant for V <= kRegKeys * kRegThreads (16384): thread t owns the
// kpt consecutive blocks [kpt t, kpt t + kpt) (kpt = V / 512 rounded up to a
// multiple of 4, at most 32) and keeps their keys in registers.
//  - Everything that reads only caller inputs (the row's position, the
//    histogram clear) happens before the wait on the logits kernel.
//  - Radix passes take 11-bit digits below the bits that the row's smallest
//    and largest keys share, into one 2048-bin shared histogram; a block scan
//    from the top bin finds the bin holding the K_b-th largest key.  Once
//    that bin holds at most 32 keys, one warp sorts them (bitonic, in
//    registers) and reads off the threshold key T and how many keys equal to
//    T are taken.
//  - The final selection is a per-thread bit mask; one block scan of
//    popcounts gives every thread the output slot of its first selected
//    block (ties go to the lower block by construction), and each thread
//    writes its selected blocks' tokens straight into the packed row.
constexpr int kRegThreads = 512;   // the launch width for many rows (two CTAs per SM)
constexpr int kRegKeys = 32;
constexpr int kDigitBits = 11;
constexpr int kBins = 1 << kDigitBits;  // 2048 = 4 bins per thread
constexpr int kTail = 32;               // a warp finishes once the chosen bin holds this few keys

template <int NWARPS>
__device__ __forceinline__ int block_sum_excl(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int x = lane < NWARPS ? scratch[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane < NWARPS) scratch[lane] = x;
  }
  __syncthreads();
  const int ex = (warp > 0 ? scratch[warp - 1] : 0) + incl - v;
  *total = scratch[NWARPS - 1];
  __syncthreads();
  return ex;
}

// KPT: keys per thread the loops are unrolled for (4, 8, 16, 24 or 32), the
// smallest that covers the launch's max_visible with CL * NT threads.
// NT: 512, or 1024 when there are fewer rows than half the SMs.
// CL: CTAs per row, one thread-block cluster (1 or 2).  With CL > 1
// the row's blocks are split in order over the cluster's CTAs; each radix
// pass sums the CTAs' shared histograms through distributed shared memory,
// so every CTA reaches the same digit, and one exchange of per-CTA counts
// places each CTA's selected blocks in the packed row.  A CTA lists its
// selected blocks in shared memory first and then expands them into their
// r tokens each with coalesced stores.
template <int KPT, int NT, int CL>
__global__ void __launch_bounds__(NT, NT == 512 && CL <= 2 ? 2 : 1) topk_reg_kernel(const TopkParams P) {
  namespace cg = cooperative_groups;
  constexpr int NW = NT / 32;
  constexpr int GT = CL * NT;  // threads per row
  __shared__ __align__(16) int hist[kBins];
  __shared__ __align__(16) int s_red[CL > 1 ? kBins : 4];  // summed bins of this CTA's slice
  __shared__ uint32_t cand[kTail];
  __shared__ int scratch[32];
  __shared__ uint32_t s_min[NW], s_max[NW];
  __shared__ int s_digit, s_k, s_cnt, s_ncand;
  __shared__ uint32_t s_cmm[2];  // this CTA's (min, max) key, read by the cluster
  __shared__ int s_ccnt[2];      // this CTA's (greater, equal) counts, read by the cluster
  constexpr int kSelCap = KPT * NT < kRegKeys * kRegThreads / 4 ? KPT * NT : kRegKeys * kRegThreads / 4;
  __shared__ int s_sel[kSelCap];  // this CTA's selected blocks in block order

  griddep_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int crank = 0;
  if constexpr (CL > 1) crank = static_cast<int>(cg::this_cluster().block_rank());
  const int row = blockIdx.x / CL;
  const int gtid = crank * NT + tid;  // thread index within the row
  // caller inputs only, before the wait
  if (crank == 0 && P.tickets != nullptr && tid < P.tickets_per_row)
    P.tickets[static_cast<long long>(row) * P.tickets_per_row + tid] = 0u;
  for (int i = tid; i < kBins; i += NT) hist[i] = 0;
  if (tid == 0) s_ncand = 0;
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
  const int kpt = min(KPT, ((V + GT - 1) / GT + 3) & ~3);
  const int base = gtid * kpt;
  int32_t* prow = P.packed + static_cast<long long>(row) * (W + 1);
  // Inside the layer step this launch also commits the row's raw key to the
  // compressor-state ring: its loads (caller inputs) are issued now, the
  // store after the wait (all pooling reads of the step are done by then).
  RingCommit rc;
  rc.slot = -1;
  const bool ring_lane = P.do_ring && crank == 0 && tid >= 32 && tid < 48;
  if (ring_lane) rc = ring_commit_prepare(P.ring, row, tid - 32);
  griddep_wait();  // logits (and, transitively, the compress kernel) are done
  if (ring_lane) ring_commit_store(P.ring, rc, tid - 32);

  const int nsel = take_all ? V : kb;
  const int tail0 = V * r;
  const int count = nsel * r + (p + 1 - tail0);
  if (!take_all) {
    // keys of blocks [base, base + kpt); 0 marks "beyond V" (no real score
    // maps to 0)
    const float* lrow = P.logits + static_cast<long long>(row) * P.ld;
    uint32_t key[KPT];
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
    for (int j = 0; j < KPT; j += 4) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (j < kpt) {
        if (base + j + 3 < V) v = *reinterpret_cast<const float4*>(lrow + base + j);
        else {
          if (base + j < V) v.x = lrow[base + j];
          if (base + j + 1 < V) v.y = lrow[base + j + 1];
          if (base + j + 2 < V) v.z = lrow[base + j + 2];
        }
      }
      const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const bool ok = j < kpt && base + j + u < V;
        key[j + u] = ok ? order_key(f[u]) : 0u;
        if (ok) {
          kmin = min(kmin, key[j + u]);
          kmax = max(kmax, key[j + u]);
        }
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, off));
      kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, off));
    }
    if (lane == 0) {
      s_min[warp] = kmin;
      s_max[warp] = kmax;
    }
    __syncthreads();
    kmin = 0xFFFFFFFFu;
    kmax = 0u;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      kmin = min(kmin, s_min[w]);
      kmax = max(kmax, s_max[w]);
    }
    if constexpr (CL > 1) {
      // the row's min and max over the cluster (this sync also orders every
      // CTA's initialisation before any remote access below)
      if (tid == 0) {
        s_cmm[0] = kmin;
        s_cmm[1] = kmax;
      }
      cg::cluster_group cluster = cg::this_cluster();
      cluster.sync();
#pragma unroll
      for (int c = 0; c < CL; ++c) {
        const uint32_t* o = cluster.map_shared_rank(s_cmm, c);
        kmin = min(kmin, o[0]);
        kmax = max(kmax, o[1]);
      }
    }
    // Bits above the highest bit where the smallest and largest keys differ
    // are common to every key: the radix passes start below them.
    const uint32_t diff = kmin ^ kmax;
    int hi = diff ? 31 - __clz(diff) : -1;
    uint32_t prefix, pmask;
    if (hi < 0) {
      prefix = kmin;
      pmask = 0xFFFFFFFFu;
    } else if (hi == 31) {
      prefix = 0u;
      pmask = 0u;
    } else {
      pmask = ~((2u << hi) - 1u);
      prefix = kmin & pmask;
    }
    int k = kb;
    while (hi >= 0) {
      const int width = hi + 1 < kDigitBits ? hi + 1 : kDigitBits;
      const int shift = hi - width + 1;
      const uint32_t dmask = (1u << width) - 1u;
      // (warp-aggregated variants -- match.any groups, or one add for a
      // warp whose keys share a bin -- measured slower or equal)
#pragma unroll
      for (int j = 0; j < KPT; ++j)
        if (key[j] != 0u && (key[j] & pmask) == prefix) atomicAdd(&hist[(key[j] >> shift) & dmask], 1);
      // bins from the top: thread t holds BPT consecutive bins
      constexpr int BPT = kBins / NT;
      int c[BPT], tot = 0;
      if constexpr (CL == 1) {
        __syncthreads();
#pragma unroll
        for (int u = 0; u < BPT; ++u) {
          c[u] = hist[kBins - 1 - BPT * tid - u];
          hist[kBins - 1 - BPT * tid - u] = 0;  // clear for a further pass
          tot += c[u];
        }
      } else {
        // The row's histogram is the sum of the cluster's CTA histograms:
        // CTA q sums bins [q S, (q + 1) S) over the cluster into its s_red
        // (16-byte remote loads), then every thread reads its four bins
        // from their owner.  Remote accesses are few and wide: distributed
        // shared memory serves them per thread, not per warp.
        static_assert(BPT == 4, "one 16-byte chunk of bins per thread");
        constexpr int S = kBins / CL;
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();  // every CTA's histogram is complete
        for (int ch = tid; ch < S / 4; ch += NT) {
          int4 acc = make_int4(0, 0, 0, 0);
#pragma unroll
          for (int q = 0; q < CL; ++q) {
            const int4 v = *reinterpret_cast<const int4*>(cluster.map_shared_rank(hist, q) + crank * S + 4 * ch);
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
          }
          *reinterpret_cast<int4*>(s_red + crank * S + 4 * ch) = acc;
        }
        cluster.sync();  // all slices are summed; no CTA reads a histogram any more
        const int b0 = kBins - BPT * (tid + 1);  // this thread's lowest bin
        const int4 v = *reinterpret_cast<const int4*>(cluster.map_shared_rank(s_red, b0 / S) + b0);
        c[0] = v.w; c[1] = v.z; c[2] = v.y; c[3] = v.x;
#pragma unroll
        for (int u = 0; u < BPT; ++u) {
          hist[kBins - 1 - BPT * tid - u] = 0;
          tot += c[u];
        }
      }
      int total;
      int cum = block_sum_excl<NW>(tot, scratch, &total);  // keys in higher bins
#pragma unroll
      for (int u = 0; u < BPT; ++u) {
        if (cum < k && k <= cum + c[u]) {
          s_digit = kBins - 1 - BPT * tid - u;
          s_k = k - cum;
          s_cnt = c[u];
        }
        cum += c[u];
      }
      __syncthreads();
      prefix |= static_cast<uint32_t>(s_digit) << shift;
      pmask |= dmask << shift;
      k = s_k;
      hi = shift - 1;
      const int cnt = s_cnt;
      if (hi >= 0 && cnt <= kTail) {
        // The chosen bin holds at most 32 keys: gather them, and one warp
        // sorts them in descending order (bitonic network over the lanes).
        // (with a cluster, all CTAs append to the first CTA's list)
        uint32_t* cl_cand = cand;
        int* cl_ncand = &s_ncand;
        if constexpr (CL > 1) {
          cl_cand = cg::this_cluster().map_shared_rank(cand, 0);
          cl_ncand = cg::this_cluster().map_shared_rank(&s_ncand, 0);
        }
#pragma unroll
        for (int j = 0; j < KPT; ++j)
          if (key[j] != 0u && (key[j] & pmask) == prefix) cl_cand[atomicAdd(cl_ncand, 1)] = key[j];
        if constexpr (CL == 1) __syncthreads();
        else cg::this_cluster().sync();
        if (warp == 0) {
          uint32_t v = lane < cnt ? cl_cand[lane] : 0u;
#pragma unroll
          for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
            for (int stride = size / 2; stride > 0; stride >>= 1) {
              const uint32_t o = __shfl_xor_sync(0xffffffffu, v, stride);
              const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
              v = keep_max ? max(v, o) : min(v, o);
            }
          }
          const uint32_t t = __shfl_sync(0xffffffffu, v, k - 1);  // k-th largest of the bin
          const int above = __popc(__ballot_sync(0xffffffffu, v > t));
          if (lane == 0) {
            s_digit = static_cast<int>(t);
            s_k = k - above;
          }
        }
        __syncthreads();
        prefix = static_cast<uint32_t>(s_digit);
        k = s_k;
        hi = -1;
      }
    }
    const uint32_t T = prefix;
    const int keq = k;
    uint32_t gt_mask = 0u, eq_mask = 0u;
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      gt_mask |= (key[j] > T ? 1u : 0u) << j;
      eq_mask |= (key[j] == T ? 1u : 0u) << j;
    }
    // one scan of (greater, equal) counts: every greater key is taken and
    // the first keq equal keys in block order
    int tot;
    const int both = block_sum_excl<NW>((__popc(gt_mask) << 16) | __popc(eq_mask), scratch, &tot);
    int gt_before = both >> 16, eq_before = both & 0xFFFF;
    int cta_gt = 0, cta_eq = 0;  // counts of the CTAs holding lower blocks
    if constexpr (CL > 1) {
      if (tid == 0) {
        s_ccnt[0] = tot >> 16;
        s_ccnt[1] = tot & 0xFFFF;
      }
      cg::cluster_group cluster = cg::this_cluster();
      cluster.sync();
      for (int c = 0; c < crank; ++c) {
        const int* o = cluster.map_shared_rank(s_ccnt, c);
        cta_gt += o[0];
        cta_eq += o[1];
      }
      gt_before += cta_gt;
      eq_before += cta_eq;
    }
    int take = keq - eq_before;
    take = take < 0 ? 0 : take;
    uint32_t eq_take = eq_mask;
    for (int c = __popc(eq_mask); c > take; --c) eq_take &= ~(1u << (31 - __clz(eq_take)));
    uint32_t m = gt_mask | eq_take;
    // this CTA's selected blocks occupy packed slots [out0, out0 + nloc)
    int out0 = 0, nloc = nsel;
    if constexpr (CL > 1) {
      out0 = cta_gt + (cta_eq < keq ? cta_eq : keq);
      int eq_loc = keq - cta_eq;
      eq_loc = eq_loc < 0 ? 0 : eq_loc > (tot & 0xFFFF) ? (tot & 0xFFFF) : eq_loc;
      nloc = (tot >> 16) + eq_loc;
    }
    int out = gt_before + (eq_before < keq ? eq_before : keq) - out0;
    while (m) {
      s_sel[out++] = base + __ffs(m) - 1;
      m &= m - 1u;
    }
    __syncthreads();
    // block b -> tokens b r .. b r + r - 1, consecutive slots of the packed row
    int32_t* dst = prow + out0 * r;
    for (int idx = tid; idx < nloc * r; idx += NT) {
      const int i = idx / r;
      dst[idx] = s_sel[i] * r + (idx - i * r);
    }
    // the tail tokens of the open group, then -1 padding
    for (int idx = nsel * r + gtid; idx < W; idx += GT)
      prow[idx] = idx < count ? tail0 + (idx - nsel * r) : -1;
    // no CTA leaves while another may still read its shared memory
    if constexpr (CL > 1) cg::this_cluster().sync();
  } else {
    for (int idx = gtid; idx < W; idx += GT) {
      int v = -1;
      if (idx < nsel * r) v = idx;  // block idx / r, token idx % r
      else if (idx < count) v = tail0 + (idx - nsel * r);
      prow[idx] = v;
    }
  }
  if (gtid == 0) prow[W] = count;
}

}  // namespace

size_t topk_smem_bytes(int max_visible, int block_topk) {
  return static_cast<size_t>(max_visible) * 4 + static_cast<size_t>(block_topk) * 4 + 16;
}

namespace {

// One cluster of CL 512-thread CTAs per row, keys per thread for max_visible.
template <int CL>
cudaError_t launch_topk_cluster(const TopkParams& p, cudaStream_t stream, bool pdl) {
  const int kpt = (p.max_visible + CL * kRegThreads - 1) / (CL * kRegThreads);
  const dim3 g(p.rows * CL), b(kRegThreads);
  if (kpt <= 4) return launch_kernel_cluster(topk_reg_kernel<4, kRegThreads, CL>, g, b, 0, stream, pdl, CL, p);
  if (kpt <= 8) return launch_kernel_cluster(topk_reg_kernel<8, kRegThreads, CL>, g, b, 0, stream, pdl, CL, p);
  return launch_kernel_cluster(topk_reg_kernel<16, kRegThreads, CL>, g, b, 0, stream, pdl, CL, p);
}

// CTAs per row for rows of more than 4096 keys: 0 = one 1024-thread CTA,
// else a cluster of that many 512-thread CTAs.  Measured on GB300: many
// rows gain from pairs while the pairs fit one wave at two CTAs per SM.
// Fewer rows run one 1024-thread CTA per row: clusters of 2, 4 or 8 per row
// were slower for the 64-row decode batch, and for the 8-row long-context
// decode four CTAs per row made about half of the replayed steps ~12 us
// slower (a two-valued step time; one CTA per row gives one value).
int topk_cluster_size(int rows, int max_visible, int sms) {
  const long long s = sms > 0 ? sms : 1;
  (void)max_visible;
  if (rows >= 76) return 2LL * rows <= 2 * s ? 2 : 1;
  return 0;
}

}  // namespace

cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream, bool pdl) {
  if (p.rows == 0) return cudaSuccess;
  if (p.max_visible <= kRegKeys * kRegThreads && p.token_topk / p.ratio <= kRegKeys * kRegThreads / 4) {
    const dim3 b(kRegThreads);
    if (p.max_visible > 4 * 1024) {
      switch (topk_cluster_size(p.rows, p.max_visible, p.sms)) {
        case 2: return launch_topk_cluster<2>(p, stream, pdl);
        case 0: {
          // one 1024-thread CTA per row, half the keys per thread
          const int kpt = (p.max_visible + 1023) / 1024;
          if (kpt <= 8) return launch_kernel(topk_reg_kernel<8, 1024, 1>, dim3(p.rows), dim3(1024), 0, stream, pdl, p);
          return launch_kernel(topk_reg_kernel<16, 1024, 1>, dim3(p.rows), dim3(1024), 0, stream, pdl, p);
        }
        default: break;
      }
    }
    const int kpt = (p.max_visible + kRegThreads - 1) / kRegThreads;
    const dim3 g(p.rows);
    if (kpt <= 4) return launch_kernel(topk_reg_kernel<4, kRegThreads, 1>, g, b, 0, stream, pdl, p);
    if (kpt <= 8) return launch_kernel(topk_reg_kernel<8, kRegThreads, 1>, g, b, 0, stream, pdl, p);
    if (kpt <= 16) return launch_kernel(topk_reg_kernel<16, kRegThreads, 1>, g, b, 0, stream, pdl, p);
    if (kpt <= 24) return launch_kernel(topk_reg_kernel<24, kRegThreads, 1>, g, b, 0, stream, pdl, p);
    return launch_kernel(topk_reg_kernel<32, kRegThreads, 1>, g, b, 0, stream, pdl, p);
  }
  const size_t smem = topk_smem_bytes(p.max_visible, p.token_topk / p.ratio);
  cudaError_t e =
      cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(topk_kernel, dim3(p.rows), dim3(kThreads), smem, stream, pdl, p);
}

}  // namespace qsa
