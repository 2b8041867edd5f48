// qsa_sparse_gqa_noalloc: the sparse GQA stage with its split-KV scratch in a
// fixed, library-owned device array instead of a caller workspace.
//
// Who needs it: callers that must not allocate device memory at the point
// where they run attention -- for example code running under an allocator
// that forbids new allocations after start-up, embedders whose memory pool is
// sized once and handed out by someone else, or plugin hosts that give a
// library only the tensors of the call.  Such callers cannot reserve the
// qsa_workspace_bytes() scratch that qsa_sparse_gqa needs for its split-KV
// partials, so this entry point keeps that scratch in a static array that is
// part of the loaded library.
//
// Costs and limits, stated for users:
//  - the array is QSA_NOALLOC_SCRATCH_BYTES (4 MiB) of device memory on
//    every GPU that loads the library, held until the process exits;
//  - a call whose split-KV partials would not fit is rejected with
//    QSA_ERR_WORKSPACE before anything is launched;
//  - every call on a device shares the one array and it keeps the last
//    call's contents; calls that may overlap on the GPU (different streams,
//    or different host threads on one device) race on it, so the caller must
//    order them (one stream, or events between streams);
//  - nothing in the array has to start at zero: every split writes all of its
//    partial outputs and log-sum-exps before the merge reads them;
//  - the first call on each device resolves the array's device address
//    (cudaGetSymbolAddress, with that device current) and caches it; make
//    that first call before any stream capture.  cudaDeviceReset unloads the
//    library's device code, so the cached address is stale afterwards: a
//    process that resets a device must not call this entry point on that
//    device again.
// Nothing here calls cudaMalloc, cudaFree or any allocating library routine.
// This entry point has no counterpart on the pages the method comes from.
#include <mutex>

#include "qsa.h"
#include "qsa_device.cuh"
#include "qsa_kernels.h"

namespace {

// The split-KV scratch.  In host code `g_noalloc_scratch` only names a
// host-side stand-in; the kernels get the device address resolved below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[QSA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
unsigned char* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device, resolved once
// per device; nullptr if the runtime refuses.
unsigned char* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
  }
  return g_scratch_ptr[dev];
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

extern "C" qsa_status qsa_sparse_gqa_noalloc(const qsa_gqa_cfg* gcfg, const void* q,
                                             const void* kv, const int32_t* block_table,
                                             int32_t bt_stride, const int32_t* packed,
                                             int32_t packed_width, const int32_t* token_to_req,
                                             const void* gate, void* out, int32_t rows,
                                             void* stream) {
  const qsa_status st = qsa::check_gcfg(gcfg);  // the checks qsa_sparse_gqa makes
  if (st != QSA_OK) return st;
  if (rows < 0) return QSA_ERR_SHAPE;
  if (rows == 0) return QSA_OK;
  if (packed_width < 2 || bt_stride < 1) return QSA_ERR_SHAPE;
  if (!q || !kv || !block_table || !packed || !token_to_req || !out) return QSA_ERR_INVALID_ARG;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kv) |
                        reinterpret_cast<uintptr_t>(gate) | reinterpret_cast<uintptr_t>(out);
  if (a16 & 15) return QSA_ERR_INVALID_ARG;

  qsa::GqaParams p{};
  p.q = static_cast<const uint16_t*>(q);
  p.kv = kv;
  p.kv_dtype = gcfg->kv_dtype;
  p.k_scale = gcfg->k_scale;
  p.v_scale = gcfg->v_scale;
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
  p.splits = qsa::gqa_num_splits(rows, gcfg->num_kv_heads, packed_width, qsa::sm_count());
  p.sms = qsa::sm_count();
  if (p.splits > 1) {
    const size_t po = static_cast<size_t>(p.splits) * rows * p.hq * 128 * sizeof(float);
    const size_t pl = static_cast<size_t>(p.splits) * rows * p.hq * sizeof(float);
    if (round256(po) + round256(pl) > QSA_NOALLOC_SCRATCH_BYTES) return QSA_ERR_WORKSPACE;
    unsigned char* scratch = scratch_on_current_device();
    if (scratch == nullptr) return QSA_ERR_CUDA;
    p.part_o = reinterpret_cast<float*>(scratch);
    p.part_lse = reinterpret_cast<float*>(scratch + round256(po));
  }
  p.err = qsa::internal_error_word();
  if (p.err == nullptr) return QSA_ERR_CUDA;
  return qsa::launch_sparse_gqa(p, static_cast<cudaStream_t>(stream), /*pdl=*/false) == cudaSuccess
             ? QSA_OK
             : QSA_ERR_CUDA;
}
