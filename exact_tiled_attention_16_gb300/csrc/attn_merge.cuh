// Exact merge of partial attention results over disjoint key sets.
//
// A partial result for key set K_s is (O_s, lse_s) with O_s normalised by its own
// sum, O_s = sum_{j in K_s} exp(s_j - lse_s) v_j and lse_s = ln sum_{j in K_s} exp(s_j).
// The result over the union is
//     lse = ln sum_s exp(lse_s),   O = sum_s exp(lse_s - lse) O_s,
// which is the running-max / running-normaliser combination the ring-attention
// page describes ("technical insight": partial results from each K/V block are
// rescaled and accumulated so that the outcome equals full attention), applied
// once per partial instead of once per block.  A partial with lse_s = -inf (no
// visible key) contributes nothing; if every partial is empty, O = 0 and
// lse = -inf.
//
// Memory-bound: each row reads S * (D + 1) floats and writes D outputs and one
// lse.  One warp per row, D/32 consecutive channels per lane (16-byte loads for
// D = 128), grid-stride over rows.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace attn {

constexpr int kMaxMergeParts = 16;

struct MergeParams {
  const float* o[kMaxMergeParts];    // partial O_s [rows, D] fp32
  const float* lse[kMaxMergeParts];  // partial lse_s [rows] fp32
  int S;
  void* out;          // [rows, D]: bf16 (out_fp32 = 0) or fp32 (may alias o[0])
  float* lse_out;     // [rows] or nullptr (may alias lse[0])
  int out_fp32;
  long long rows;
};

template <int D>
__global__ void __launch_bounds__(256) attn_merge_kernel(const MergeParams mp) {
  constexpr int kPer = D / 32;  // channels per lane
  const int lane = threadIdx.x & 31;
  const long long warp_global = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long r = warp_global; r < mp.rows; r += nwarps) {
    float m = -INFINITY;
    for (int s = 0; s < mp.S; ++s) m = fmaxf(m, __ldg(mp.lse[s] + r));
    float acc[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
    float z = 0.f;
    if (m != -INFINITY) {
      for (int s = 0; s < mp.S; ++s) {
        const float w = expf(__ldg(mp.lse[s] + r) - m);
        z += w;
        const float* src = mp.o[s] + r * D + lane * kPer;
        if constexpr (kPer == 4) {
          const float4 x = *reinterpret_cast<const float4*>(src);
          acc[0] += w * x.x;
          acc[1] += w * x.y;
          acc[2] += w * x.z;
          acc[3] += w * x.w;
        } else {
#pragma unroll
          for (int i = 0; i < kPer; ++i) acc[i] += w * src[i];
        }
      }
    }
    const float inv_z = z > 0.f ? 1.f / z : 0.f;
    const float lse = z > 0.f ? m + logf(z) : -INFINITY;
    if (mp.out_fp32) {
      float* dst = static_cast<float*>(mp.out) + r * D + lane * kPer;
#pragma unroll
      for (int i = 0; i < kPer; ++i) dst[i] = acc[i] * inv_z;
    } else {
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(mp.out) + r * D + lane * kPer;
#pragma unroll
      for (int i = 0; i < kPer; i += 2) {
        __nv_bfloat162 h = __floats2bfloat162_rn(acc[i] * inv_z, acc[i + 1] * inv_z);
        *reinterpret_cast<__nv_bfloat162*>(dst + i) = h;
      }
    }
    if (mp.lse_out != nullptr && lane == 0) mp.lse_out[r] = lse;
  }
}

}  // namespace attn
