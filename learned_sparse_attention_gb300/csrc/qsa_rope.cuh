// Indexer query / key preparation shared by the compress and logits kernels:
// Gemma RMSNorm, NeoX rotation of dims 0..63 (1-D or interleaved 3-section
// MRoPE) and the cos|sin table lookup, one half-warp per 128-dim vector,
// 8 consecutive dims per lane.
//
// Follows "vllm.models.qwen4_exp.nvidia.qsa", QSAIndexer.forward (unfused
// path: gemma_rmsnorm -> apply_qsa_rope -> cast) and "indexer_qsa.py",
// apply_qsa_rope (NeoX pairs (i, i + rotary_dim/2), cos|sin halves of the
// caller's table, interleaved MRoPE sections).
#pragma once

#include "qsa_device.cuh"
#include "qsa_kernels.h"

namespace qsa {

struct RopeParams {
  const float* cos_sin;  // [max_pos, 64]: cos of the 32 frequencies, then sin
  int max_pos, mrope, sec_h, sec_w;
  unsigned long long* err;
};

__device__ __forceinline__ RopeParams rope_params(const CompressParams& P) {
  return RopeParams{P.cos_sin, P.max_pos, P.mrope, P.sec_h, P.sec_w, P.err};
}

// Interleaved MRoPE: frequency i uses the H component if i % 3 == 1 and
// i < 3 * sec_h, W if i % 3 == 2 and i < 3 * sec_w, T otherwise.
__device__ __forceinline__ int mrope_component(int i, int mrope, int sec_h, int sec_w) {
  if (!mrope) return 0;
  if (i % 3 == 1 && i < 3 * sec_h) return 1;
  if (i % 3 == 2 && i < 3 * sec_w) return 2;
  return 0;
}

__device__ __forceinline__ void load8_bf16(const uint16_t* src, float (&x)[8]) {
  const uint4 v = *reinterpret_cast<const uint4*>(src);
  x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x);
  x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
  x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z);
  x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
}

// cos/sin of the 8 frequencies this lane touches, at a 3-component position.
__device__ __forceinline__ void rope_coeffs(const RopeParams& P, int lane16,
                                            const int64_t (&pos)[3], float (&c)[8],
                                            float (&s)[8]) {
  const int fbase = 8 * (lane16 & 3);
  if (!P.mrope) {
    int64_t pp = pos[0];
    if (pp < 0 || pp >= P.max_pos) {
      if (lane16 == 0) flag_error(P.err);
      pp = pp < 0 ? 0 : P.max_pos - 1;
    }
    const float4* row = reinterpret_cast<const float4*>(P.cos_sin + pp * 64 + fbase);
    const float4 c0 = row[0], c1 = row[1], s0 = row[8], s1 = row[9];
    c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w; c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
    s[0] = s0.x; s[1] = s0.y; s[2] = s0.z; s[3] = s0.w; s[4] = s1.x; s[5] = s1.y; s[6] = s1.z; s[7] = s1.w;
    return;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int i = fbase + e;
    // (a select, not an index: pos stays in registers)
    const int comp = mrope_component(i, P.mrope, P.sec_h, P.sec_w);
    int64_t pp = comp == 0 ? pos[0] : comp == 1 ? pos[1] : pos[2];
    if (pp < 0 || pp >= P.max_pos) {
      if (lane16 == 0 && e == 0) flag_error(P.err);
      pp = pp < 0 ? 0 : P.max_pos - 1;
    }
    const float* row = P.cos_sin + pp * 64;
    c[e] = row[i];
    s[e] = row[32 + i];
  }
}

// Gemma RMSNorm over the half-warp's 128 dims, then NeoX rotation of dims
// 0..63, in place on x (this lane's 8 dims).
__device__ __forceinline__ void norm_rope(float (&x)[8], const float (&w1)[8], float eps,
                                          int lane16, const float (&c)[8], const float (&s)[8]) {
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
  for (int off = 8; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float inv = rsqrtf(ss * (1.0f / 128) + eps);
#pragma unroll
  for (int e = 0; e < 8; ++e) x[e] = x[e] * inv * w1[e];
  float partner[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) partner[e] = __shfl_xor_sync(0xffffffffu, x[e], 4);
  if (lane16 < 4) {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = x[e] * c[e] - partner[e] * s[e];
  } else if (lane16 < 8) {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = x[e] * c[e] + partner[e] * s[e];
  }
}

}  // namespace qsa
