// Block-level pieces shared by several kernels of the layer step so that small
// jobs ride along in a neighbouring launch instead of a launch of their own:
// the ring commit (stage 1 bookkeeping, done by the top-k launch) and the
// row group of each logits CTA.
#pragma once

#include "qsa_device.cuh"
#include "qsa_kernels.h"

namespace qsa {

// Ring commit of one row by 16 lanes: the row's raw key (and 3-D position)
// goes to ring slot p % S of its request, unless a later row of the same
// request in this step maps to the same slot.  Must run after every pooling
// read of the step.  Split in two so that the loads (caller inputs only) can
// run before a kernel waits on its predecessor and only the store after.
struct RingCommit {
  long long slot;  // ring row, or -1 for no write
  uint4 key;       // this lane's 16 bytes of the raw key
  long long pos;   // this lane's position component (lanes 0-2, MRoPE)
};

__device__ __forceinline__ RingCommit ring_commit_prepare(const CompressParams& P, int row,
                                                          int lane16) {
  RingCommit rc;
  rc.slot = -1;
  rc.pos = 0;
  const int req = P.token_to_req[row];
  if (req < 0 || req >= P.reqs) return rc;  // counted by the compress kernel
  const int last_row = P.qsl[req + 1] - 1;
  if (last_row < row || last_row >= P.rows) {  // inconsistent query_start_loc
    if (lane16 == 0) flag_error(P.err);
    return rc;
  }
  const int p = P.logical[row];
  const int p_last = P.logical[last_row];
  if (p + P.S <= p_last) return rc;  // overwritten later in this step
  const int ring_block = P.ring_bt[static_cast<long long>(req) * P.ring_bt_stride];
  if (ring_block < 0 || ring_block >= P.ring_blocks || p < 0) {
    if (lane16 == 0) flag_error(P.err);
    return rc;
  }
  rc.slot = static_cast<long long>(ring_block) * P.S + (p % P.S);
  rc.key = *reinterpret_cast<const uint4*>(P.raw_keys + static_cast<long long>(row) * 128 + 8 * lane16);
  if (P.ring_pos != nullptr && lane16 < 3) rc.pos = P.positions[static_cast<long long>(row) * 3 + lane16];
  return rc;
}

__device__ __forceinline__ void ring_commit_store(const CompressParams& P, const RingCommit& rc,
                                                  int lane16) {
  if (rc.slot < 0) return;
  *reinterpret_cast<uint4*>(P.ring + rc.slot * 128 + 8 * lane16) = rc.key;
  if (P.ring_pos != nullptr && lane16 < 3) P.ring_pos[rc.slot * 3 + lane16] = rc.pos;
}

__device__ __forceinline__ void ring_commit_row(const CompressParams& P, int row, int lane16) {
  ring_commit_store(P, ring_commit_prepare(P, row, lane16), lane16);
}

// Row group g of the logits kernel, found by the whole block: the rows of
// each request in chunks of R, numbered in request order.  Returns
// (row0, nrows, request, 0), or row0 = -1 when g is past the last group.
__device__ __forceinline__ int4 find_group(const int32_t* qsl, int reqs, int rows, int R, int g,
                                           unsigned long long* err) {
  __shared__ int warp_tot[32];
  __shared__ int carry;
  __shared__ int4 found;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  if (tid == 0) {
    carry = 0;
    found = make_int4(-1, 0, 0, 0);
  }
  __syncthreads();
  for (int base = 0; base < reqs; base += blockDim.x) {
    const int q = base + tid;
    int n = 0, start = 0;
    if (q < reqs) {
      start = qsl[q];
      n = qsl[q + 1] - start;
      if (n < 0 || start < 0 || start + n > rows) {  // rows outside [0, rows): skipped
        if (g == 0) flag_error(err);
        n = 0;
      }
    }
    const int ng = (n + R - 1) / R;
    int incl = ng;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int v = lane < nwarps ? warp_tot[lane] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += y;
      }
      if (lane < nwarps) warp_tot[lane] = v;
    }
    __syncthreads();
    const int excl = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + incl - ng;
    if (q < reqs && g >= excl && g < excl + ng) {
      const int k = g - excl;
      found = make_int4(start + k * R, min(R, n - k * R), q, 0);
    }
    __syncthreads();
    if (tid == 0) carry += warp_tot[nwarps - 1];
    const bool done = found.x >= 0;
    __syncthreads();
    if (done) break;
  }
  return found;
}

// The L-th (row, key chunk) item that holds keys, for one row per group:
// row r has ceil(ceil(vis(r) / 128) / tpc) chunks (vis(r) = its visible
// compressed keys), items numbered row-major; found by the whole block.
// Returns (row, chunk, 0, 0), or row = -1 when L is past the last item.
__device__ __forceinline__ int4 find_row_chunk(const int32_t* logical, int rows, int ratio,
                                               int tpc, int L) {
  __shared__ int warp_tot[32];
  __shared__ int carry;
  __shared__ int4 found;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  if (tid == 0) {
    carry = 0;
    found = make_int4(-1, 0, 0, 0);
  }
  __syncthreads();
  for (int base = 0; base < rows; base += blockDim.x) {
    const int r = base + tid;
    int nc = 0;
    if (r < rows) {
      const int p = logical[r];
      const int vis = p < 0 ? 0 : (p + 1) / ratio;
      nc = ((vis + 127) / 128 + tpc - 1) / tpc;
    }
    int incl = nc;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int v = lane < nwarps ? warp_tot[lane] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += y;
      }
      if (lane < nwarps) warp_tot[lane] = v;
    }
    __syncthreads();
    const int excl = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + incl - nc;
    if (r < rows && L >= excl && L < excl + nc) found = make_int4(r, L - excl, 0, 0);
    __syncthreads();
    if (tid == 0) carry += warp_tot[nwarps - 1];
    const bool done = found.x >= 0;
    __syncthreads();
    if (done) break;
  }
  return found;
}

}  // namespace qsa
