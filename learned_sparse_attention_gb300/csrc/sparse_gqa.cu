// Stage 4 of the QSA layer step: sparse paged GQA over the selected tokens.
//
// Follows "vllm.models.qwen4_exp.nvidia.ops.qsa", qsa_sparse_paged_attention
// (packed selection buffer whose trailing column is the loop bound, paged
// K/V through the block table of the row's request, split-KV partials in
// fp32 merged by log-sum-exp, mandatory output gate) and the patch's
// _qsa_sparse_paged_gqa_splitk_kernel (score scale D^-1/2 in the exp2
// domain, invalid entries masked, output divided by the normaliser and zero
// when nothing is valid, bf16 rounding of the attention output before the
// sigmoid gate).
//
// GB300 mapping.  Decode is an HBM gather: every selected token costs 512
// contiguous bytes (K then V of one KV head).  One CTA = (row, KV head,
// split), 4 warps.  Each warp owns 16 tokens of every 64-token tile and runs
// its own cp.async ring over them (16-byte copies, one token row per warp
// instruction, XOR-swizzled so ldmatrix is conflict-free); each tile's
// copies are issued before the previous tile is computed.  The GQA
// group of query heads is the N = 8 side of m16n8k16 MMAs with the tokens
// on M (groups of 1 to 8 heads fill one column block, zero queries in the
// unused columns; groups of 16 take two blocks that share every K and V
// fragment):
//   S^T[16 tok x 8 heads] = K[16 x 128] . Q^T          (8 k-steps)
//   O^T[128 dims x 8 heads] += V^T[128 x 16] . P^T       (8 m-tiles)
// P^T comes from the S^T accumulator with one movmatrix transpose per 8x8
// block; each lane keeps the online-softmax state of its two heads, the same
// heads its O^T fragments hold.  The state's reference max moves only when a
// score passes it by a margin, so most slabs skip the max reduction and the
// rescale.  The four warps are merged in shared memory.  Launches of many
// waves with four KV heads (a prefill chunk) take one CTA per row instead:
// warp w runs KV head w over all the row's tokens in the same way and
// finishes its own heads, with no merge.
// A prologue resolves the CTA's token range (packed index -> block table ->
// KV row id, in chunks of up to 2560 tokens) into shared memory in parallel,
// so the copy issue of a slab never waits on a dependent global load; the
// inputs that do not depend on the top-k kernel (q, gate, the request's
// block-table row) are loaded before the dependency wait, and the first
// chunk's packed entries together with the count right after it.  CTAs run
// in KV-head-major order.  With split-KV, the last CTA
// of a (row, KV head) to finish merges the fp32 partials (an atomic ticket
// per (row, KV head)), so no second launch is needed when a ticket array is
// given.
#include "qsa_device.cuh"
#include "qsa_kernels.h"
#include "qsa_launch.cuh"

namespace qsa {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kRidBatch = 8;  // KV row ids resolved per thread per batch
constexpr int kFirst = 20;    // packed entries per thread loaded right after the wait
constexpr int kTile = 64;      // tokens per CTA tile (16 per warp)
constexpr int kMaxTiles = 40;                // tiles of one row-id chunk
constexpr int kMaxTok = kMaxTiles * kTile;   // token row ids staged at a time
constexpr uint32_t kBadRow = 0xFFFFFFFFu;

// Shared-memory plan per KV dtype (KVT 0: bf16, 1: e4m3) and ring depth
// ST.  A warp's stage holds its 16 tokens' K rows, then their V rows, in
// 16-byte chunks XOR-swizzled by token.  e4m3 rows are half as wide, so the
// ring is deeper at the same footprint.  bf16 runs 3 stages at two CTAs
// per SM when the launch is about one wave (HBM latency to hide), 2 stages
// at three CTAs per SM when it is many waves (prefill: K/V mostly from L2,
// and more warps to issue).
template <int KVT, int ST>
struct KvPlan {
  static constexpr int kRowB = KVT ? 256 : 512;          // K|V bytes of one (token, KV head)
  static constexpr int kStages = ST;
  static constexpr int kSlab = 16 * kRowB;                // bytes per warp stage
  static constexpr int kPipe = kWarps * kStages * kSlab;
  static constexpr int kSmem = kPipe + kMaxTok * 4;
};
constexpr float kLog2e = 1.4426950408889634f;
// 2^x by the PTX approximate base-2 exponential, subnormal results flushed
// to zero (softmax weights that small do not register next to the others).
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// A head's softmax reference moves only when a score passes it by more than
// this (log2 units): the exponentials stay <= 256, well inside bf16 / f16.
constexpr float kLazy = 8.0f;

__device__ __forceinline__ float sigmoidf_(float g) { return 1.0f / (1.0f + __expf(-g)); }

// The gate of 8 dims (bf16x8), or zeros when there is none.
__device__ __forceinline__ uint4 load_gate8(const GqaParams& P, long long obase) {
  return P.gate != nullptr ? *reinterpret_cast<const uint4*>(P.gate + obase) : make_uint4(0, 0, 0, 0);
}

// out[8 dims] = bf16(bf16(x) * sigmoid(gate)) (or bf16(x) without a gate).
__device__ __forceinline__ void store_out8(const GqaParams& P, long long obase, const float (&x)[8],
                                           uint4 gr) {
  const float gv[8] = {bf16_lo(gr.x), bf16_hi(gr.x), bf16_lo(gr.y), bf16_hi(gr.y),
                       bf16_lo(gr.z), bf16_hi(gr.z), bf16_lo(gr.w), bf16_hi(gr.w)};
  float y[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    y[e] = bf16_round(x[e]);
    if (P.gate != nullptr) y[e] = y[e] * sigmoidf_(gv[e]);
  }
  uint4 ov;
  ov.x = pack_bf16x2(y[0], y[1]);
  ov.y = pack_bf16x2(y[2], y[3]);
  ov.z = pack_bf16x2(y[4], y[5]);
  ov.w = pack_bf16x2(y[6], y[7]);
  *reinterpret_cast<uint4*>(P.out + obase) = ov;
}

// Log-sum-exp merge of the split partials of 8 dims of one (row, head).
__device__ __forceinline__ void merge8(const GqaParams& P, int row, int hq, int d0, uint4 gr) {
  float M = -INFINITY;
  for (int s = 0; s < P.splits; ++s)
    M = fmaxf(M, __ldcg(P.part_lse + (static_cast<long long>(s) * P.rows + row) * P.hq + hq));
  float W = 0.f, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s < P.splits; ++s) {
    const long long pb = (static_cast<long long>(s) * P.rows + row) * P.hq + hq;
    const float lse = __ldcg(P.part_lse + pb);
    if (lse == -INFINITY) continue;
    const float wt = exp2f(lse - M);
    W += wt;
    const float4* po = reinterpret_cast<const float4*>(P.part_o + pb * 128 + d0);
    const float4 a = __ldcg(po), b = __ldcg(po + 1);
    acc[0] += wt * a.x; acc[1] += wt * a.y; acc[2] += wt * a.z; acc[3] += wt * a.w;
    acc[4] += wt * b.x; acc[5] += wt * b.y; acc[6] += wt * b.z; acc[7] += wt * b.w;
  }
  const float inv = W > 0.f ? 1.0f / W : 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] *= inv;
  store_out8(P, (static_cast<long long>(row) * P.hq + hq) * 128 + d0, acc, gr);
}

// KV row id (block * Hkv + kvh) * page + offset of a selected token, or
// kBadRow for a masked entry (a block id outside the cache).  The host
// rejects caches whose row ids would not fit 32 bits.
__device__ __forceinline__ uint32_t kv_row_id(const GqaParams& P, int off, int pid, int kvh) {
  if (pid < 0 || pid >= P.num_blocks) return kBadRow;
  return (static_cast<uint32_t>(pid) * P.hkv + kvh) * static_cast<uint32_t>(P.page) + off;
}

// NB: column blocks of 8 query heads (1 for groups of 1-8, 2 for 16).
// KVT: KV cache dtype, 0 bf16, 1 e4m3 with static scales (f16 MMAs: every
// e4m3 value and every bf16 query of normal range is exact in f16).
// ROW: one CTA per row, warp w taking KV head w over all the row's tokens
// (four KV heads, no split): the row's selection is resolved once for its
// four KV heads and each warp finishes its own heads, with no merge across
// warps.  Used for launches of many waves, where a CTA's fixed costs
// (resolving the selection, the ring's fill and drain, the merge) weigh.
template <int NB, int KVT, int ST, bool ROW>
__global__ void __launch_bounds__(kThreads) gqa_kernel(const GqaParams P) {
  static_assert(!ROW || (NB == 1 && KVT == 0), "row CTAs: bf16 KV, groups of up to 8 heads");
  using KP = KvPlan<KVT, ST>;
  constexpr int kStages = KP::kStages;
  constexpr int kSlab = KP::kSlab;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint32_t s_vmask[kWarps][kStages];
  __shared__ int s_last;
  uint32_t* s_rowid = reinterpret_cast<uint32_t*>(smem + KP::kPipe);
  const uint8_t* kvb = static_cast<const uint8_t*>(P.kv);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // KV-head-major CTA order: the CTAs resident at one time mostly share a
  // KV head, so the rows of a request that select the same tokens (prefill
  // chunks, speculative rows) find them in L2
  const int kvh = ROW ? warp : static_cast<int>(blockIdx.x) / P.rows;
  const int row = ROW ? static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x) - kvh * P.rows;
  const int pair = row * P.hkv + kvh;  // merge ticket of this (row, KV head)
  const int split = blockIdx.y;
  // row CTAs resolve KV head 0's row ids; warp w's rows are page * w further
  const uint8_t* kvw = kvb + (ROW ? static_cast<long long>(warp) * P.page * KP::kRowB : 0ll);
  const int g = lane >> 2, t = lane & 3;
  const int Wcols = P.packed_width - 1;

  const int G = P.group;
  griddep_launch_dependents();
  const int req = P.token_to_req[row];
  const int32_t* prow = P.packed + static_cast<long long>(row) * P.packed_width;
  // Q^T fragments (B operand of S^T = K.Q^T): head kvh * G + 8 nb + g (zero
  // past the group), 2 dims per register; a caller input, loaded before
  // waiting for the top-k kernel (after it when the same layer step's
  // main-attention prepare writes q and the gate).
  uint32_t qb[NB][8][2];
  auto load_q = [&]() {
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    const int hl = nb * 8 + g;
    const uint16_t* qh = P.q + (static_cast<long long>(row) * P.hq + kvh * G + min(hl, G - 1)) * 128;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      if (KVT == 0) {
        qb[nb][kk][0] = hl < G ? *reinterpret_cast<const uint32_t*>(qh + 16 * kk + 2 * t) : 0u;
        qb[nb][kk][1] = hl < G ? *reinterpret_cast<const uint32_t*>(qh + 16 * kk + 8 + 2 * t) : 0u;
      } else {
        // f16 B fragments over the same dimension order as the decoded e4m3
        // K fragments: k-step kk pairs (2t, 2t+1) <- dims 16 kk + 4t + {0, 1}
        // and (2t+8, 2t+9) <- dims 16 kk + 4t + {2, 3}
        const uint2 v = hl < G ? *reinterpret_cast<const uint2*>(qh + 16 * kk + 4 * t) : make_uint2(0u, 0u);
        qb[nb][kk][0] = bf16x2_to_f16x2(v.x);
        qb[nb][kk][1] = bf16x2_to_f16x2(v.y);
      }
    }
  }
  };
  // The request's block-table row (a caller input) is copied before the
  // wait into the last pipeline stage of all warps (contiguous, and not
  // written before the main loop), so that resolving the selected tokens'
  // pages after the wait costs shared-memory reads.  Longer rows, and
  // token ranges of more than one chunk, read the table in global memory.
  const int32_t* bt_row = P.block_table + static_cast<long long>(req < 0 ? 0 : req) * P.bt_stride;
  int32_t* s_bt = reinterpret_cast<int32_t*>(smem + (kStages - 1) * kWarps * kSlab);
  const bool bt_fits = P.bt_stride <= kWarps * kSlab / 4;
  const float vscale = KVT ? P.v_scale : 1.0f;
  if (bt_fits) {
    for (int i0 = threadIdx.x; i0 < P.bt_stride; i0 += 8 * kThreads) {
      int v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = i0 + u * kThreads < P.bt_stride ? bt_row[i0 + u * kThreads] : 0;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (i0 + u * kThreads < P.bt_stride) s_bt[i0 + u * kThreads] = v[u];
    }
  }
  // the epilogue's items of this thread, 8 dims each, and their gate (a
  // caller input): item tid + 128 i is head item / 16 of the group; with row
  // CTAs a warp finishes its own 8 heads, lane + 32 i being head item / 16
  constexpr int NI = ROW ? 4 : NB;
  const int d0 = (threadIdx.x & 15) * 8;
  uint4 gate8[NI];
  auto load_gates = [&]() {
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int hh = ROW ? (lane + 32 * i) >> 4 : (threadIdx.x + kThreads * i) >> 4;
      gate8[i] = hh < G ? load_gate8(P, (static_cast<long long>(row) * P.hq + kvh * G + hh) * 128 + d0)
                        : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  if (!P.q_after_wait) {
    load_q();
    load_gates();
  }
  griddep_wait();  // the packed selection (and merge tickets) are written
  if (P.q_after_wait) {
    load_q();
    load_gates();
  }
  // Without split-KV the CTA's range starts at token 0 whatever the count,
  // so its first entries (kFirst per thread, up to kFirst * kThreads tokens)
  // load together with the count: one round trip before the first copies.
  int tk[kFirst];
#pragma unroll
  for (int u = 0; u < kFirst; ++u) {
    const int i = threadIdx.x + u * kThreads;
    tk[u] = (P.splits == 1 && i < Wcols) ? prow[i] : -1;
  }
  int n = prow[Wcols];
  bool bad_row = req < 0;
  if (n < 0 || n > Wcols) {
    bad_row = true;
    n = 0;
  }
  if (bad_row) {
    n = 0;
    if (threadIdx.x == 0) flag_error(P.err);
  }
  const int ntiles = (n + kTile - 1) / kTile;
  const int tps = (ntiles + P.splits - 1) / P.splits;
  const int tb = split * tps;
  const int te = min(ntiles, tb + tps);
  const int tok0 = tb * kTile;
  const int ntok = te > tb ? min(te * kTile, n) - tok0 : 0;
  const int32_t* ptok = prow + tok0;
  const bool sbt = bt_fits && ntok <= kMaxTok;
  __syncthreads();  // the staged block-table row is complete

  float o[NB][8][4];
  float m0[NB], m1[NB], l0[NB], l1[NB];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[nb][mt][0] = o[nb][mt][1] = o[nb][mt][2] = o[nb][mt][3] = 0.f;
    m0[nb] = m1[nb] = -INFINITY;
    l0[nb] = l1[nb] = 0.f;
  }
  // 128^-0.5 * log2(e), and the static K scale of an e4m3 cache folded in
  const float sl2 = 0.08838834764831845f * kLog2e * (KVT ? P.k_scale : 1.0f);
  bool bad = false;

  // KV row ids of the selected tokens tok[u] (u < NT) into
  // s_rowid[i0 + u * kThreads]; entries at or past cn are not touched.
  // (pages are a power of two in practice: shift and mask instead of a
  // division there)
  const bool page_pow2 = (P.page & (P.page - 1)) == 0;
  const int page_shift = __ffs(P.page) - 1;
  auto resolve = [&](auto& tok, int i0, int cn) {
    constexpr int NT = sizeof(tok) / sizeof(tok[0]);
    int pid[NT], off[NT];
#pragma unroll
    for (int u = 0; u < NT; ++u) {
      const int blk = tok[u] < 0 ? -1 : page_pow2 ? tok[u] >> page_shift : tok[u] / P.page;
      off[u] = tok[u] - blk * P.page;
      pid[u] = -1;
      if (tok[u] >= 0 && blk < P.bt_stride) pid[u] = sbt ? s_bt[blk] : bt_row[blk];
    }
#pragma unroll
    for (int u = 0; u < NT; ++u) {
      const int i = i0 + u * kThreads;
      if (i >= cn) continue;
      const uint32_t rid = kv_row_id(P, off[u], pid[u], ROW ? 0 : kvh);
      bad |= rid == kBadRow;
      s_rowid[i] = rid;
    }
  };
  // The first kFirst entries per thread of the first chunk.
  {
    const int cn = min(kMaxTok, ntok);
#pragma unroll
    for (int u = 0; u < kFirst; ++u) {
      const int i = threadIdx.x + u * kThreads;
      if (i >= cn) tk[u] = -1;
      else if (P.splits != 1) tk[u] = ptok[i];
    }
    resolve(tk, threadIdx.x, cn);
  }

  // The range runs in chunks of at most kMaxTok tokens whose KV row ids are
  // resolved into shared memory (in batches of kRidBatch loads per thread)
  // before the chunk's copies start.
  for (int c0 = 0; c0 < ntok; c0 += kMaxTok) {
    const int cn = min(kMaxTok, ntok - c0);
    const int nt = ROW ? (cn + 15) / 16 : (cn + kTile - 1) / kTile;  // slabs of this warp
    if (c0 > 0) __syncthreads();  // every warp has issued the previous chunk's copies
    const int i_begin = c0 == 0 ? kFirst * kThreads : 0;
    for (int i0 = i_begin + threadIdx.x; i0 < cn; i0 += kRidBatch * kThreads) {
      int tok[kRidBatch];
#pragma unroll
      for (int u = 0; u < kRidBatch; ++u) {
        const int i = i0 + u * kThreads;
        tok[u] = i < cn ? ptok[c0 + i] : -1;
      }
      resolve(tok, i0, cn);
    }
    __syncthreads();  // all row ids of the chunk are resolved

    auto issue = [&](int tile, int stage) {
      const int li = (ROW ? tile * 16 : tile * kTile + warp * 16) + (lane & 15);
      const uint32_t rid = (lane < 16 && li < cn) ? s_rowid[li] : kBadRow;
      const uint32_t vm = __ballot_sync(0xffffffffu, rid != kBadRow) & 0xffffu;
      if (lane == 0) s_vmask[warp][stage] = vm;
      uint8_t* dst_base = smem + (stage * kWarps + warp) * kSlab;
      if (KVT == 0) {  // one 512-byte row per instruction
        const int chunk = lane & 15, is_v = lane >> 4;
        const uint8_t* src_lane = kvw + is_v * 256 + chunk * 16;
        if (vm == 0xFFFFu) {  // a full slab (the common case): no per-row masks
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const uint32_t rj = __shfl_sync(0xffffffffu, rid, j);
            cp_async16_full(dst_base + is_v * 4096 + j * 256 + ((chunk ^ (j & 7)) << 4),
                            src_lane + static_cast<long long>(rj) * 512);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const uint32_t rj = __shfl_sync(0xffffffffu, rid, j);
            const bool okj = (vm >> j) & 1u;
            uint8_t* dst = dst_base + is_v * 4096 + j * 256 + ((chunk ^ (j & 7)) << 4);
            cp_async16(dst, src_lane + static_cast<long long>(okj ? rj : 0u) * 512, okj ? 16u : 0u);
          }
        }
      } else {  // two 256-byte rows per instruction
        const int chunk = lane & 7, is_v = (lane >> 3) & 1, sub = lane >> 4;
        const uint8_t* src_lane = kvw + is_v * 128 + chunk * 16;
        if (vm == 0xFFFFu) {
#pragma unroll
          for (int j2 = 0; j2 < 8; ++j2) {
            const int j = 2 * j2 + sub;
            const uint32_t rj = __shfl_sync(0xffffffffu, rid, j);
            cp_async16_full(dst_base + is_v * 2048 + j * 128 + ((chunk ^ (j & 7)) << 4),
                            src_lane + static_cast<long long>(rj) * 256);
          }
        } else {
#pragma unroll
          for (int j2 = 0; j2 < 8; ++j2) {
            const int j = 2 * j2 + sub;
            const uint32_t rj = __shfl_sync(0xffffffffu, rid, j);
            const bool okj = (vm >> j) & 1u;
            uint8_t* dst = dst_base + is_v * 2048 + j * 128 + ((chunk ^ (j & 7)) << 4);
            cp_async16(dst, src_lane + static_cast<long long>(okj ? rj : 0u) * 256, okj ? 16u : 0u);
          }
        }
      }
    };

#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
      if (s < nt) issue(s, s);
      cp_async_commit();
    }
    for (int it = 0; it < nt; ++it) {
      cp_async_wait<kStages - 2>();
      // tile it has landed for every lane, and every lane is done with tile
      // it - 1, whose stage takes the next copies now: they overlap this
      // tile's compute
      __syncwarp();
      {
        const int nxt = it + kStages - 1;
        if (nxt < nt) issue(nxt, nxt % kStages);
        cp_async_commit();
      }
      const int stage = it % kStages;
      const uint8_t* sK = smem + (stage * kWarps + warp) * kSlab;
      const uint8_t* sV = sK + 8 * KP::kRowB;
      // S^T = K.Q^T over 8 K-steps, split over two accumulators so that the
      // MMAs form two dependent chains of four instead of one of eight (each
      // K fragment feeds every column block)
      float sa[NB][2][4];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int c = 0; c < 2; ++c) sa[nb][c][0] = sa[nb][c][1] = sa[nb][c][2] = sa[nb][c][3] = 0.f;
      if (KVT == 0) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          uint32_t a[4];
          const int rl = lane & 15;
          const int ch = 2 * kk + (lane >> 4);
          ldmatrix_x4(a, sK + rl * 256 + ((ch ^ (rl & 7)) << 4));
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) mma_bf16_16816(sa[nb][kk & 1], a, qb[nb][kk][0], qb[nb][kk][1]);
        }
      } else {
        // one ldmatrix.x4 brings 32 e4m3 dims of the warp's 16 rows: per lane
        // dims 4t..4t+3 of rows g and g+8 for two 16-dim k-steps, decoded to
        // the f16 A fragments in the order the query fragments use
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
          uint32_t a[4];
          const int rl = lane & 15;
          const int ch = 2 * k2 + (lane >> 4);
          ldmatrix_x4(a, sK + rl * 128 + ((ch ^ (rl & 7)) << 4));
          uint32_t fa[4], fb[4];
          e4m3x4_to_f16x2x2(a[0], fa[0], fa[2]);
          e4m3x4_to_f16x2x2(a[1], fa[1], fa[3]);
          e4m3x4_to_f16x2x2(a[2], fb[0], fb[2]);
          e4m3x4_to_f16x2x2(a[3], fb[1], fb[3]);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            mma_f16_16816(sa[nb][0], fa, qb[nb][2 * k2][0], qb[nb][2 * k2][1]);
            mma_f16_16816(sa[nb][1], fb, qb[nb][2 * k2 + 1][0], qb[nb][2 * k2 + 1][1]);
          }
        }
      }
      const uint32_t vm = s_vmask[warp][stage];
      const bool v0 = (vm >> g) & 1u, v1 = (vm >> (g + 8)) & 1u;
      uint32_t pb[NB][2];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        float sc[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[e] = sa[nb][0][e] + sa[nb][1][e];
        // m0 / m1 are each head's reference for the exponentials, not its
        // exact running max: they move (with the max reduction over the
        // warp and the rescale of the sums and the accumulator) only when
        // some score exceeds its head's reference by more than kLazy, so
        // every p stays <= 2^kLazy; m, l and o stay consistent with one
        // another, which is all the merges and the final division use.
        // y: the exponent of each entry (token g / g+8, head 2t / 2t+1)
        // against its head's reference, +inf while a head has none yet,
        // -inf for the tokens of a partial slab that are not selected.
        float y[4] = {fmaf(sc[0], sl2, -m0[nb]), fmaf(sc[1], sl2, -m1[nb]), fmaf(sc[2], sl2, -m0[nb]),
                      fmaf(sc[3], sl2, -m1[nb])};
        if (vm != 0xFFFFu) {
          if (!v0) y[0] = y[1] = -INFINITY;
          if (!v1) y[2] = y[3] = -INFINITY;
        }
        const bool up = fmaxf(fmaxf(y[0], y[1]), fmaxf(y[2], y[3])) > kLazy;
        if (__any_sync(0xffffffffu, up)) {
          float mx0 = fmaxf(v0 ? sc[0] : -INFINITY, v1 ? sc[2] : -INFINITY) * sl2;
          float mx1 = fmaxf(v0 ? sc[1] : -INFINITY, v1 ? sc[3] : -INFINITY) * sl2;
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
          }
          const float mn0 = fmaxf(m0[nb], mx0), mn1 = fmaxf(m1[nb], mx1);
          const float al0 = ex2_ftz(m0[nb] - (mn0 == -INFINITY ? 0.f : mn0));
          const float al1 = ex2_ftz(m1[nb] - (mn1 == -INFINITY ? 0.f : mn1));
          l0[nb] *= al0;
          l1[nb] *= al1;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            o[nb][mt][0] *= al0;
            o[nb][mt][1] *= al1;
            o[nb][mt][2] *= al0;
            o[nb][mt][3] *= al1;
          }
          m0[nb] = mn0;
          m1[nb] = mn1;
          y[0] = v0 ? fmaf(sc[0], sl2, -mn0) : -INFINITY;
          y[1] = v0 ? fmaf(sc[1], sl2, -mn1) : -INFINITY;
          y[2] = v1 ? fmaf(sc[2], sl2, -mn0) : -INFINITY;
          y[3] = v1 ? fmaf(sc[3], sl2, -mn1) : -INFINITY;
        }
        const float p0 = ex2_ftz(y[0]), p1 = ex2_ftz(y[1]);
        const float p2 = ex2_ftz(y[2]), p3 = ex2_ftz(y[3]);
        l0[nb] += p0 + p2;
        l1[nb] += p1 + p3;
        pb[nb][0] = movmatrix_trans(KVT ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1));
        pb[nb][1] = movmatrix_trans(KVT ? pack_f16x2(p2, p3) : pack_bf16x2(p2, p3));
      }
      if (KVT == 0) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t a[4];
          const int tk = (lane & 7) + ((lane >> 4) << 3);
          const int ch = 2 * mt + ((lane >> 3) & 1);
          ldmatrix_x4_trans(a, sV + tk * 256 + ((ch ^ (tk & 7)) << 4));
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) mma_bf16_16816(o[nb][mt], a, pb[nb][0], pb[nb][1]);
        }
      } else {
        // V^T fragments straight from the e4m3 rows: m-tiles 2P and 2P + 1
        // take dims 32P + 4g + {0, 1} and {2, 3} in their rows g and g + 8,
        // so one 32-bit load per token gives a lane its four dims; byte
        // permutes pair tokens (2t, 2t+1) and (2t+8, 2t+9) per dim before
        // the e4m3 -> f16 conversion
#pragma unroll
        for (int P2 = 0; P2 < 4; ++P2) {
          const int c = 2 * P2 + (g >> 2);  // 16-byte chunk of dims 32 P2 + 4 g
          const int bo = (g & 3) * 4;
          uint32_t w[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int tk = 2 * t + (u & 1) + ((u >> 1) << 3);
            w[u] = *reinterpret_cast<const uint32_t*>(sV + tk * 128 + ((c ^ (tk & 7)) << 4) + bo);
          }
          uint32_t a0[4], a1[4];  // m-tiles 2 P2 and 2 P2 + 1
          e4m3x4_to_f16x2x2(prmt(w[0], w[1], 0x5140u), a0[0], a0[1]);
          e4m3x4_to_f16x2x2(prmt(w[0], w[1], 0x7362u), a1[0], a1[1]);
          e4m3x4_to_f16x2x2(prmt(w[2], w[3], 0x5140u), a0[2], a0[3]);
          e4m3x4_to_f16x2x2(prmt(w[2], w[3], 0x7362u), a1[2], a1[3]);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            mma_f16_16816(o[nb][2 * P2], a0, pb[nb][0], pb[nb][1]);
            mma_f16_16816(o[nb][2 * P2 + 1], a1, pb[nb][0], pb[nb][1]);
          }
        }
      }
    }
    cp_async_wait<0>();
  }
  if (bad) flag_error(P.err);

  if constexpr (ROW) {
    // the warp's 8 heads, normalised, through its own first ring stage (its
    // copies have all landed) to 16-byte stores with the gate
    __syncwarp();
    float* co = reinterpret_cast<float*>(smem + warp * kSlab);  // [8 heads][128 dims]
    float la = l0[0], lb = l1[0];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      la += __shfl_xor_sync(0xffffffffu, la, off);
      lb += __shfl_xor_sync(0xffffffffu, lb, off);
    }
    const float ia = la > 0.f ? 1.0f / la : 0.f, ib = lb > 0.f ? 1.0f / lb : 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int d = 16 * mt + g;  // accumulator rows g and g + 8 of m-tile mt
      co[(2 * t) * 128 + d] = o[0][mt][0] * ia;
      co[(2 * t + 1) * 128 + d] = o[0][mt][1] * ib;
      co[(2 * t) * 128 + d + 8] = o[0][mt][2] * ia;
      co[(2 * t + 1) * 128 + d + 8] = o[0][mt][3] * ib;
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int hh = (lane + 32 * i) >> 4;
      if (hh >= G) continue;
      const float4 a = *reinterpret_cast<const float4*>(co + hh * 128 + d0);
      const float4 b = *reinterpret_cast<const float4*>(co + hh * 128 + d0 + 4);
      const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      store_out8(P, (static_cast<long long>(row) * P.hq + kvh * G + hh) * 128 + d0, x, gate8[i]);
    }
    return;
  }

  __syncthreads();  // pipeline buffers are free from here on
  float* cm = reinterpret_cast<float*>(smem);   // [warps][8 NB] max
  float* cl = cm + kWarps * 8 * NB;             // [warps][8 NB] sum
  float* co = cl + kWarps * 8 * NB;             // [warps][8 NB heads][128 dims]
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    float la = l0[nb], lb = l1[nb];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      la += __shfl_xor_sync(0xffffffffu, la, off);
      lb += __shfl_xor_sync(0xffffffffu, lb, off);
    }
    const int hb = warp * 8 * NB + nb * 8;
    if (lane < 4) {
      cm[hb + 2 * t] = m0[nb];
      cm[hb + 2 * t + 1] = m1[nb];
      cl[hb + 2 * t] = la;
      cl[hb + 2 * t + 1] = lb;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      // accumulator rows g and g + 8 of m-tile mt -> dims d and d + dd
      const int d = KVT ? 32 * (mt >> 1) + 4 * g + 2 * (mt & 1) : 16 * mt + g;
      const int dd = KVT ? 1 : 8;
      co[(hb + 2 * t) * 128 + d] = o[nb][mt][0];
      co[(hb + 2 * t + 1) * 128 + d] = o[nb][mt][1];
      co[(hb + 2 * t) * 128 + d + dd] = o[nb][mt][2];
      co[(hb + 2 * t + 1) * 128 + d + dd] = o[nb][mt][3];
    }
  }
  __syncthreads();

#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    const int hh = (threadIdx.x + kThreads * nb) >> 4;  // head within the group
    if (hh >= G) continue;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, cm[w * 8 * NB + hh]);
    float L = 0.f, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = cm[w * 8 * NB + hh];
      const float wt = mw == -INFINITY ? 0.f : exp2f(mw - M);
      L += cl[w * 8 * NB + hh] * wt;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += co[(w * 8 * NB + hh) * 128 + d0 + e] * wt;
    }
    // the static V scale of an e4m3 cache multiplies the normalised output
    // (and every split partial alike: the merge is linear in them)
    const float inv = L > 0.f ? vscale / L : 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] *= inv;
    const int hq = kvh * G + hh;
    if (P.splits == 1) {
      store_out8(P, (static_cast<long long>(row) * P.hq + hq) * 128 + d0, acc, gate8[nb]);
      continue;
    }
    const long long pb = (static_cast<long long>(split) * P.rows + row) * P.hq + hq;
    float4* po = reinterpret_cast<float4*>(P.part_o + pb * 128 + d0);
    po[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    po[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    if ((threadIdx.x & 15) == 0) P.part_lse[pb] = L > 0.f ? M + __log2f(L) : -INFINITY;
  }
  if (P.splits == 1) return;
  if (P.counters == nullptr) return;  // a separate merge launch follows
  // The last split of this (row, KV head) to finish merges them all.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(P.counters + pair, 1u);
    s_last = prev == static_cast<unsigned>(P.splits - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    const int hh = (threadIdx.x + kThreads * nb) >> 4;
    if (hh < G) merge8(P, row, kvh * G + hh, d0, gate8[nb]);
  }
  if (threadIdx.x == 0) P.counters[pair] = 0u;  // ready for the next launch
}

// Log-sum-exp merge of the split partials, then bf16 rounding and the gate.
__global__ void __launch_bounds__(256) gqa_merge_kernel(const GqaParams P) {
  griddep_launch_dependents();
  griddep_wait();  // all split partials are written
  const int row = blockIdx.x;
  for (int idx = threadIdx.x; idx < P.hq * 16; idx += blockDim.x) {
    const int hq = idx >> 4, d0 = (idx & 15) * 8;
    merge8(P, row, hq, d0, load_gate8(P, (static_cast<long long>(row) * P.hq + hq) * 128 + d0));
  }
}

}  // namespace

// Split-KV count: about two CTAs per SM, and no CTA with more than kMaxTiles
// 64-token tiles (one chunk of staged row ids, so that the request's
// block-table row is read from shared memory).
int gqa_num_splits(int rows, int hkv, int packed_width, int sms) {
  const long long base = static_cast<long long>(rows) * hkv;
  if (base <= 0) return 1;
  const int max_tiles = (packed_width - 1 + kTile - 1) / kTile;
  const int min_s = (max_tiles + kMaxTiles - 1) / kMaxTiles;
  // as many splits as keep every (row, KV head, split) CTA resident in one
  // wave at two CTAs per SM (shared memory): a CTA's time grows with its
  // tokens, so shorter splits finish the launch sooner
  long long s = 2ll * sms / base;
  if (s > max_tiles) s = max_tiles;
  if (s > 64) s = 64;
  if (s < min_s) s = min_s;
  if (s < 1) s = 1;
  return static_cast<int>(s);
}

cudaError_t launch_sparse_gqa(const GqaParams& p, cudaStream_t stream, bool pdl,
                              bool zero_tickets) {
  if (p.rows == 0) return cudaSuccess;
  if (static_cast<long long>(p.num_blocks) * p.hkv * p.page >= static_cast<long long>(kBadRow))
    return cudaErrorInvalidValue;
  if (p.group < 1 || (p.group > 8 && p.group != 16)) return cudaErrorInvalidValue;
  if (p.kv_dtype != 0 && p.kv_dtype != 1) return cudaErrorInvalidValue;
  // kernels by [column blocks][ring plan: bf16 3 stages, bf16 2 stages,
  // e4m3 5 stages, bf16 2 stages with row CTAs]
  void (*kerns[2][4])(const GqaParams) = {
      {gqa_kernel<1, 0, 3, false>, gqa_kernel<1, 0, 2, false>, gqa_kernel<1, 1, 5, false>,
       gqa_kernel<1, 0, 2, true>},
      {gqa_kernel<2, 0, 3, false>, gqa_kernel<2, 0, 2, false>, gqa_kernel<2, 1, 5, false>,
       gqa_kernel<2, 0, 2, false>}};
  const int smems[4] = {KvPlan<0, 3>::kSmem, KvPlan<0, 2>::kSmem, KvPlan<1, 5>::kSmem,
                        KvPlan<0, 2>::kSmem};
  const int ki = p.group <= 8 ? 0 : 1;
  const long long ctas = static_cast<long long>(p.rows) * p.hkv * p.splits;
  const bool many = ctas > 4ll * (p.sms > 0 ? p.sms : 1);
  int plan = p.kv_dtype == 1 ? 2 : many ? 1 : 0;
  if (plan == 1 && ki == 0 && p.hkv == kWarps && p.splits == 1) plan = 3;
  auto kern = kerns[ki][plan];
  const int kSmem = smems[plan];
  static bool attr_set[2][4][64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[ki][plan][dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[ki][plan][dev] = true;
  }
  if (p.splits > 1 && p.counters != nullptr && zero_tickets) {
    cudaError_t e = cudaMemsetAsync(p.counters, 0, sizeof(unsigned) * p.rows * p.hkv, stream);
    if (e != cudaSuccess) return e;
    pdl = false;  // a memset node sits between this kernel and its predecessor
  }
  const dim3 grid = plan == 3 ? dim3(p.rows, 1) : dim3(p.rows * p.hkv, p.splits);
  cudaError_t e = launch_kernel(kern, grid, dim3(kThreads), kSmem, stream, pdl, p);
  if (e != cudaSuccess || p.splits == 1 || p.counters != nullptr) return e;
  return launch_kernel(gqa_merge_kernel, dim3(p.rows), dim3(256), 0, stream, true, p);
}

}  // namespace qsa
