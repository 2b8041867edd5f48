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
//   warp 0      allocates TMEM, loads the B tile with one TMA box and issues
//               tcgen05.mma (one thread) into two accumulator buffers so the
//               epilogue overlaps the next tile;
//   warps 1-4   A-tile producers, through a ring of 3 (N <= 64) to 8 stages.
//               The keys of a tile sit on 128 / cpage scattered compressed
//               pages (2 KB each for e4m3 and 16-key pages).  For pages of 8
//               or more keys, warp 1 loads them with one TMA box per page
//               (SW128, completing on the stage's mbarrier), one lane per
//               box so the boxes of a tile are in flight together: the
//               gather then leaves the SM's load/store pipe to the
//               epilogue's stores.  Shorter pages use 16-byte cp.async
//               straight into the swizzled layout (lanes on whole key rows
//               for e4m3 at N <= 64, one key row per thread otherwise);
//   warps 5..   epilogue: one wide tcgen05.ld of the accumulator, branch-free
//               ReLU / head sums, scale, coalesced fp32 stores.
// Every wait is bounded (see mbar_wait); a timeout sets the error word.
#include "qsa_device.cuh"
#include "qsa_kernels.h"
#include "qsa_launch.cuh"
#include "stage_helpers.cuh"

namespace qsa {
namespace {

// G: row groups per CTA.  With G = 2 a CTA runs two row groups of the same
// request over one stream of key tiles: each A tile feeds two MMAs (one per
// group, into the two TMEM accumulators in turn), which halves the A-tile
// traffic per FLOP; the epilogue of one group overlaps the other group's MMA.
// TMA: the A tiles come by TMA (one producer warp) rather than cp.async (four).
template <int IDT, int NPAD, int G = 1, bool TMA = false>
struct LogitsCfg {
  static constexpr int ATOMS = IDT == 1 ? 1 : 2;        // 128-byte K atoms per key row
  static constexpr int A_ATOM = 128 * 128;              // bytes of one atom of a 128-key tile
  static constexpr int A_STAGE = A_ATOM * ATOMS;
  static constexpr int B_ATOM = NPAD * 128;
  static constexpr int B_GROUP = B_ATOM * ATOMS;        // one row group's query tile
  static constexpr int B_BYTES = B_GROUP * G;
  static constexpr int MAX_ROWS = 64;                   // rows per CTA (G * rows per group)
  static constexpr int MAX_PAGES = 4096;                // page ids staged per CTA (at most)
  // decode-sized tiles (N <= 64) keep 3 stages so that 4 CTAs fit on an SM;
  // from N = 128 on a CTA has the SM to itself (TMEM, registers), and the A
  // ring takes what shared memory is left after B and the page ids (at most
  // 8 stages): the A tiles come from L2 and need many bytes in flight.
  static constexpr int SMEM_LIMIT = 226 * 1024;  // 227 KB per CTA, less static smem
  static constexpr int STAGES_FIT =
      (SMEM_LIMIT - 1024 - B_BYTES - 256 - MAX_ROWS * 4 - MAX_PAGES * 4) / A_STAGE;
  static constexpr int STAGES = NPAD <= 64 ? 3 : (STAGES_FIT < 8 ? STAGES_FIT : 8);
  // from N = 128 on one epilogue warpgroup per 64 accumulator columns: the
  // ReLU + head sums are chains of dependent adds, and only several warps
  // per scheduler hide their latency behind the MMA of the next tile
  static constexpr int EPI_WG = NPAD >= 128 ? NPAD / 64 : 1;
  static constexpr int TEAMS = EPI_WG >= 2 ? 2 : 1;     // epilogue teams taking items in turn
  static constexpr int PRODUCERS = TMA ? 32 : 128;      // producer threads (cp.async: a key row each)
  // Copy mapping of the A gather.  Lanes on whole key rows (every fetched
  // 32-byte sector used in full) measured faster for e4m3 keys streamed from
  // HBM at N <= 64 (decode); one key row per thread measured faster for bf16
  // keys and for the L2-resident keys of long prefill row groups.
  static constexpr bool COALESCED = IDT == 1 && NPAD <= 64;
  static constexpr int THREADS = 32 + PRODUCERS + 128 * EPI_WG;
  static constexpr int KSTEPS = IDT == 1 ? 4 : 8;       // 32 bytes of K per MMA
  static constexpr uint32_t TMEM_COLS = 2 * NPAD;
  // shared memory without the page-id array, which is sized per launch
  static constexpr int SMEM_BASE = 1024 + STAGES * A_STAGE + B_BYTES + 256 + MAX_ROWS * 4;
  static_assert(STAGES >= 3 && SMEM_BASE + MAX_PAGES * 4 <= SMEM_LIMIT, "shared memory");
};

template <int IDT, int NPAD, int G, bool TMA>
__global__ void __launch_bounds__(LogitsCfg<IDT, NPAD, G, TMA>::THREADS, 1)
    index_logits_kernel(const __grid_constant__ CUtensorMap tmap_q,
                        const __grid_constant__ CUtensorMap tmap_cc, const LogitsParams P) {
  using C = LogitsCfg<IDT, NPAD, G, TMA>;
  griddep_launch_dependents();
  // Everything up to griddep_wait reads only caller inputs (metadata, page
  // tables), so it overlaps the tail of the compress kernel.
  const int R = P.rows_per_group;
  int4 grp;
  int chunk = blockIdx.y;
  bool remapped = false;
  if constexpr (NPAD <= 64) {  // (compiled into the narrow kernels only)
    if (P.remap) {  // one row per group: the L-th item that holds keys
      const int L = blockIdx.y * gridDim.x + blockIdx.x;
      const int4 rc = find_row_chunk(P.logical, P.rows, P.ratio, P.tiles_per_cta, L);
      grp = make_int4(rc.x, 1, rc.x >= 0 ? P.token_to_req[rc.x] : 0, 0);
      chunk = rc.y;
      if (rc.x >= 0 && (grp.z < 0 || grp.z >= P.reqs)) {
        if (threadIdx.x == 0) flag_error(P.err);
        grp.x = -1;
      }
      remapped = true;
    }
  }
  // Wide kernels (prefill-sized row groups) take the groups last-first: the
  // later groups of a causal chunk see more keys, so the longest CTAs start
  // in the first wave and the last wave holds the shortest ones.
  const int gidx = NPAD >= 128 ? static_cast<int>(gridDim.x - 1 - blockIdx.x) : static_cast<int>(blockIdx.x);
  if (!remapped) grp = find_group(P.qsl, P.reqs, P.rows, R * G, gidx, P.err);
  // The kernels after this one rely on "logits complete" implying "compress
  // complete", so CTA (0, 0) waits for the compress kernel even when it has
  // no work (the other idle CTAs leave at once and free their slots).
  const bool keeps_order = blockIdx.x == 0 && blockIdx.y == 0;
  if (grp.x < 0) {
    if (keeps_order) griddep_wait();
    return;
  }
  const int row0 = grp.x, nrows = grp.y, req = grp.z;
  const int p_last = P.logical[row0 + nrows - 1];
  const int vmax = p_last < 0 ? 0 : (p_last + 1) / P.ratio;
  const int total_tiles = (vmax + 127) / 128;
  const int t_begin = chunk * P.tiles_per_cta;
  const int t_end = min(total_tiles, t_begin + P.tiles_per_cta);
  if (t_begin >= t_end) {
    if (keeps_order) griddep_wait();
    return;
  }
  const int ntiles = t_end - t_begin;
  const int ngroups = (nrows + R - 1) / R;  // row groups in this CTA (<= G)
  const int nitems = ntiles * ngroups;      // work item j: key tile j / ngroups, group j % ngroups

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
  int* s_vis = reinterpret_cast<int*>(smem_raw + pad + C::STAGES * C::A_STAGE + C::B_BYTES + 256);
  int* s_page = s_vis + C::MAX_ROWS;  // tiles_per_cta * (128 / cpage) entries

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cpage = P.cpage;
  const int32_t* bt_row = P.cblock_table + static_cast<long long>(req) * P.cbt_stride;
  // Prologue: the group's visible-block counts and the physical compressed
  // pages of this CTA's key range (-1: beyond the group's keys, -2: an
  // out-of-range page id, counted and read as zeros), resolved in parallel.
  const int ppt = 128 / cpage;  // pages per 128-key tile
  const int page0 = t_begin * ppt;
  const int npages = ntiles * ppt;  // <= tiles_per_cta * ppt <= MAX_PAGES (host)
  const int last_page = (vmax - 1) / cpage;
  for (int i = threadIdx.x; i < npages; i += blockDim.x) {
    const int lp = page0 + i;
    int phys = -1;
    if (lp <= last_page && lp < P.cbt_stride) {
      phys = bt_row[lp];
      if (phys < 0 || phys >= P.cpages) {
        flag_error(P.err);
        phys = -2;
      }
    }
    s_page[i] = phys;
  }
  for (int r = threadIdx.x; r < nrows; r += blockDim.x) {
    const int pr = P.logical[row0 + r];
    s_vis[r] = pr < 0 ? 0 : (pr + 1) / P.ratio;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], TMA ? 1 : C::PRODUCERS);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 4 * (C::EPI_WG / C::TEAMS));  // one arrival per warp of a team
    }
    mbar_init(bar_q, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  unsigned long long* err = P.err;
  // The TMA producer waits later, after issuing the tiles that hold no key
  // this step's compress kernel can write; every other warp waits here.
  if (!(TMA && warp == 1)) griddep_wait();  // the query tile and this step's compressed keys are written

  if (warp == 0) {
    // ------------------------------------------------------ B tile + MMA issuer
    if (lane == 0) {
      tma_prefetch_desc(&tmap_q);
      if (TMA) tma_prefetch_desc(&tmap_cc);
      mbar_arrive_expect_tx(bar_q, ngroups * C::B_GROUP);
      for (int g = 0; g < ngroups; ++g) {
#pragma unroll
        for (int atom = 0; atom < C::ATOMS; ++atom)
          tma_load_2d(sB + g * C::B_GROUP + atom * C::B_ATOM, &tmap_q, atom * 64,
                      (row0 + g * R) * P.n_heads, bar_q);
      }
      uint32_t idesc[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const int rows_g = min(R, nrows - g * R);
        uint32_t n_eff = ((max(rows_g, 1) * P.n_heads + 31) / 32) * 32;
        if (n_eff > NPAD) n_eff = NPAD;
        idesc[g] = umma_idesc(IDT == 1 ? 0u : 1u, 128, n_eff);
      }
      bool ok = mbar_wait(bar_q, 0, err);
      // smem descriptors: the start-address field (address / 16, 14 bits)
      // takes byte offsets / 16 without carrying out (shared memory < 256 KB)
      const uint64_t a_desc0 = umma_sdesc_sw128(smem_addr(sA));
      const uint64_t b_desc0 = umma_sdesc_sw128(smem_addr(sB));
      int g = 0, s = 0;
      uint32_t ph = 0;
      for (int j = 0; ok && j < nitems; ++j) {
        const int a = j & 1;
        const uint32_t aph = (j >> 1) & 1;
        if (!mbar_wait(&acc_empty[a], aph ^ 1, err)) break;
        if (g == 0 && !mbar_wait(&full[s], ph, err)) break;
        tc_fence_after_sync();
        const uint64_t a_desc = a_desc0 + ((s * C::A_STAGE) >> 4);
        const uint64_t b_desc = b_desc0 + ((g * C::B_GROUP) >> 4);
        const uint32_t d_tmem = tmem_base + a * NPAD;
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {
          const uint32_t off = (kk & 3) * 32;  // byte offset inside a 128-byte K atom
          const uint64_t adesc = a_desc + (((kk >> 2) * C::A_ATOM + off) >> 4);
          const uint64_t bdesc = b_desc + (((kk >> 2) * C::B_ATOM + off) >> 4);
          const uint32_t id = (G == 1 || g == 0) ? idesc[0] : idesc[G - 1];
          if (IDT == 1)
            umma_f8f6f4(d_tmem, adesc, bdesc, id, kk > 0 ? 1u : 0u);
          else
            umma_f16(d_tmem, adesc, bdesc, id, kk > 0 ? 1u : 0u);
        }
        if (g == ngroups - 1) umma_commit(&empty[s]);  // the tile's last reader
        umma_commit(&acc_full[a]);
        if (++g == ngroups) {  // next key tile
          g = 0;
          if (++s == C::STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (TMA && warp == 1) {
    // ------------------------------------------------------ A tiles by TMA
    // Warp 1: box b of a tile = page b % ppt, 128-byte K atom b / ppt.  Lane
    // 0 arms the stage's barrier with the bytes of the valid boxes, then
    // every lane issues its box.  Pages past the group's keys are skipped
    // (those rows are never stored); an out-of-range page id is read as
    // zeros, written before the barrier is armed.
    //
    // The compress kernel of this step writes only the compressed keys of
    // groups that hold one of this step's tokens: for a request whose first
    // new token is at position f (its rows are consecutive positions), keys
    // below floor(f / ratio) are caller inputs.  The ring's first tiles
    // made only of such keys are issued before the dependency wait, so
    // their gather overlaps the compress kernel.
    if (warp == 1) {
      const int nbox = C::ATOMS * ppt;  // <= 32 for cpage >= 8
      const uint32_t box_bytes = static_cast<uint32_t>(cpage) * 128u;
      const int elems_per_atom = 128 / (IDT == 1 ? 1 : 2);
      const int f = min(P.logical[P.qsl[req]], P.logical[row0]);
      const int c_safe = f < 0 ? 0 : f / P.ratio;
      const int n_early = max(0, min(min(ntiles, C::STAGES), c_safe / 128 - t_begin));
      if (n_early == 0) griddep_wait();
      for (int i = 0; i < ntiles; ++i) {
        if (i == n_early && n_early > 0) griddep_wait();
        const int s = i % C::STAGES;
        const uint32_t ph = (i / C::STAGES) & 1;
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&empty[s], ph ^ 1, err);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        const int j = lane % ppt, atom = lane / ppt;
        const int phys = lane < nbox ? s_page[i * ppt + j] : -1;
        uint8_t* dst = sA + s * C::A_STAGE + atom * C::A_ATOM + j * cpage * 128;
        if (phys == -2) {
          for (uint32_t o = 0; o < box_bytes; o += 16)
            *reinterpret_cast<uint4*>(dst + o) = make_uint4(0u, 0u, 0u, 0u);
          fence_proxy_async_smem();
        }
        const unsigned valid = __ballot_sync(0xffffffffu, phys >= 0);
        if (lane == 0) mbar_arrive_expect_tx(&full[s], __popc(valid) * box_bytes);
        __syncwarp();
        if (phys >= 0) tma_load_2d(dst, &tmap_cc, atom * elems_per_atom, phys * cpage, &full[s]);
      }
    }
  } else if (!TMA && warp <= C::PRODUCERS / 32) {
    // ------------------------------------------------------ A-tile producers
    // Thread m copies key row m of every tile: 8 (e4m3) or 16 (bf16) 16-byte
    // cp.async into the 128-byte-swizzled K-major layout the MMA reads.  A
    // tile is announced (proxy fence + arrive) once LAG newer tiles are in
    // flight, so LAG + 1 tiles stream at a time.
    constexpr int LAG = C::STAGES - 2;
    constexpr int CH = 8 * C::ATOMS;
    const int m = threadIdx.x - 32;
    int issued = 0;
    for (int i = 0; i < ntiles; ++i) {
      const int s = i % C::STAGES;
      const uint32_t ph = (i / C::STAGES) & 1;
      if (!mbar_wait(&empty[s], ph ^ 1, err)) break;
      if constexpr (!C::COALESCED) {
        const int key = (t_begin + i) * 128 + m;
        const int phys = s_page[min(i * ppt + m / cpage, npages - 1)];
        const bool ok = key < vmax && phys >= 0;
        const uint8_t* src = P.ccache + (static_cast<long long>(ok ? phys : 0) * cpage + (m % cpage)) *
                                            P.row_bytes;
        uint8_t* dst = sA + s * C::A_STAGE + m * 128;
#pragma unroll
        for (int c = 0; c < CH; ++c)
          cp_async16(dst + (c >> 3) * C::A_ATOM + (((c & 7) ^ (m & 7)) << 4), src + c * 16,
                     ok ? 16u : 0u);
      } else {
        // step c copies 16-byte chunk m % CH of key row c * (128 / CH) + m / CH:
        // CH consecutive lanes cover one whole key row, so every 32-byte sector
        // a warp fetches is used in full
        const int chunk = m % CH;
        uint8_t* dst0 = sA + s * C::A_STAGE + (chunk >> 3) * C::A_ATOM;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int row = c * (128 / CH) + m / CH;
          const int key = (t_begin + i) * 128 + row;
          const int phys = s_page[min(i * ppt + row / cpage, npages - 1)];
          const bool ok = key < vmax && phys >= 0;
          const uint8_t* src = P.ccache +
                               (static_cast<long long>(ok ? phys : 0) * cpage + (row % cpage)) * P.row_bytes +
                               chunk * 16;
          cp_async16(dst0 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4), src, ok ? 16u : 0u);
        }
      }
      cp_async_commit();
      ++issued;
      if (i >= LAG) {
        cp_async_wait<LAG>();
        fence_proxy_async_smem();
        mbar_arrive(&full[(i - LAG) % C::STAGES]);
      }
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    for (int i = max(0, issued - LAG); i < issued; ++i) mbar_arrive(&full[i % C::STAGES]);
  } else {
    // ------------------------------------------------------------ epilogue
    // The epilogue warpgroups form C::TEAMS teams that take the items in
    // turn: team t handles items t, t + TEAMS, ...  With two teams each team
    // owns one TMEM accumulator (and, with two row groups per CTA, one
    // group), so one team's wait for its next accumulator overlaps the other
    // team's work.
    constexpr int WGT = C::EPI_WG / C::TEAMS;  // warpgroups per team
    constexpr int COLS = NPAD / WGT;           // accumulator columns of a warpgroup
    constexpr int NSEG = COLS / 8;
    const int wg = (warp - 1 - C::PRODUCERS / 32) >> 2;
    const int team = wg / WGT;
    const int lane_base = 32 * (warp & 3);
    const int m = lane_base + lane;
    const int col_begin = (wg % WGT) * COLS;
    const int r0 = col_begin / P.n_heads;
    // the row group of this team's items (two teams, two groups: team t has
    // group t; otherwise every item is group 0)
    const int gq = (C::TEAMS == 2 && ngroups == 2) ? team : 0;
    const int rows_g = min(R, nrows - gq * R);
    const int nlive = max(0, min(rows_g * P.n_heads, col_begin + COLS) - col_begin) / P.n_heads;
    const int* vis = s_vis + gq * R + r0;
    float* const out0 = P.logits + static_cast<long long>(row0 + gq * R + r0) * P.ld;
    for (int j = team; j < nitems; j += C::TEAMS) {
      const int a = j & 1;
      const uint32_t aph = (j >> 1) & 1;
      const int i = ngroups == 2 ? (j >> 1) : j;  // key tile of item j
      if (!mbar_wait(&acc_full[a], aph, err)) break;
      tc_fence_after_sync();
      const int key = (t_begin + i) * 128 + m;
      // The warpgroup's columns in 32-column TMEM reads (the other epilogue
      // warps hide each read's latency).  relu(x) is summed as x + |x| (one
      // FMA-pipe add with an absolute-value operand; the factor 1/2 is folded
      // into the scale) over pairs added with packed f32x2 adds.  Measured:
      // max(x, 0) on the ALU pipe saturated it beside the MMA-issuing warp's
      // integer work, and scalar add chains starved that warp of issue slots.
      // The accumulator goes straight back to the MMA warp, then the head sums
      // (packed pairs, one final add per row) and the stores follow.
      constexpr int NCH = COLS / 32;
      unsigned long long seg[NSEG];
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(lane_base) << 16) + a * NPAD + col_begin;
#pragma unroll
      for (int h = 0; h < NCH; ++h) {
        uint32_t x[32];
        tmem_ld32_issue(taddr + h * 32, x);
        tmem_wait_ld32(x);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          unsigned long long pr[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x0 = __uint_as_float(x[q * 8 + 2 * e]);
            const float x1 = __uint_as_float(x[q * 8 + 2 * e + 1]);
            pr[e] = f32x2_pack(x0 + fabsf(x0), x1 + fabsf(x1));  // 2 relu(x)
          }
          seg[h * 4 + q] = f32x2_add(f32x2_add(pr[0], pr[1]), f32x2_add(pr[2], pr[3]));
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_relaxed(&acc_empty[a]);
      // pairwise tree up to n_heads columns per row (n_heads is 8, 16, 32
      // or 64): branch-free, compact.
      if (P.n_heads >= 16) {
#pragma unroll
        for (int q = 0; q < NSEG / 2; ++q) seg[q] = f32x2_add(seg[2 * q], seg[2 * q + 1]);
      }
      if (P.n_heads >= 32) {
#pragma unroll
        for (int q = 0; q < NSEG / 4; ++q) seg[q] = f32x2_add(seg[2 * q], seg[2 * q + 1]);
      }
      if (P.n_heads >= 64) {
#pragma unroll
        for (int q = 0; q < NSEG / 8; ++q) seg[q] = f32x2_add(seg[2 * q], seg[2 * q + 1]);
      }
#pragma unroll
      for (int q = 0; q < NSEG; ++q) {
        if (q >= nlive) break;  // uniform across the warpgroup
        if (key < vis[q]) out0[q * P.ld + key] = f32x2_hsum(seg[q]) * (0.5f * P.scale);
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <int IDT, int NPAD, int G, bool TMA>
cudaError_t launch_cfg(const LogitsParams& p, const CUtensorMap& tq, const CUtensorMap& tcc,
                       int max_groups, int chunks, cudaStream_t stream, bool pdl) {
  using C = LogitsCfg<IDT, NPAD, G, TMA>;
  auto kern = index_logits_kernel<IDT, NPAD, G, TMA>;
  const int smem = C::SMEM_BASE + p.tiles_per_cta * (128 / p.cpage) * 4;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BASE + C::MAX_PAGES * 4);
    if (e != cudaSuccess) return e;
    // all of the unified L1 / shared memory as shared memory, so that as many
    // CTAs as the shared-memory footprint allows are resident on an SM
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  return launch_kernel(kern, dim3(max_groups, chunks), dim3(C::THREADS), smem, stream, pdl, tq, tcc,
                       p);
}

template <int IDT, int NPAD>
cudaError_t launch_one(const LogitsParams& p, const CUtensorMap& tq, const CUtensorMap& tcc,
                       int max_groups, int chunks, cudaStream_t stream, bool pdl) {
  if (!p.tma_a) return launch_cfg<IDT, NPAD, 1, false>(p, tq, tcc, max_groups, chunks, stream, pdl);
  if constexpr (IDT == 1 && NPAD == 256) {
    if (p.groups_per_cta == 2)
      return launch_cfg<IDT, NPAD, 2, true>(p, tq, tcc, max_groups, chunks, stream, pdl);
  }
  return launch_cfg<IDT, NPAD, 1, true>(p, tq, tcc, max_groups, chunks, stream, pdl);
}

}  // namespace

cudaError_t launch_index_logits(const LogitsParams& p, const CUtensorMap& tq,
                                const CUtensorMap& tcc, int index_dtype, int npad,
                                int max_groups, int chunks, cudaStream_t stream, bool pdl) {
  if (max_groups <= 0 || chunks <= 0) return cudaSuccess;
  if (index_dtype == 1) {
    switch (npad) {
      case 32: return launch_one<1, 32>(p, tq, tcc, max_groups, chunks, stream, pdl);
      case 64: return launch_one<1, 64>(p, tq, tcc, max_groups, chunks, stream, pdl);
      case 128: return launch_one<1, 128>(p, tq, tcc, max_groups, chunks, stream, pdl);
      case 256: return launch_one<1, 256>(p, tq, tcc, max_groups, chunks, stream, pdl);
    }
  } else {
    switch (npad) {
      case 32: return launch_one<0, 32>(p, tq, tcc, max_groups, chunks, stream, pdl);
      case 64: return launch_one<0, 64>(p, tq, tcc, max_groups, chunks, stream, pdl);
      case 128: return launch_one<0, 128>(p, tq, tcc, max_groups, chunks, stream, pdl);
      case 256: return launch_one<0, 256>(p, tq, tcc, max_groups, chunks, stream, pdl);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace qsa
