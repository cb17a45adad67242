// Diagnostics of the library.
//  * The two ways the softmax can take its exponentials -- ex2.approx on the
//    special-function unit and the FMA-pipe polynomial exp2_poly2 -- evaluated on
//    caller data (for tests against the host's exact 2^x) and timed on the device
//    the caller has current.  The benchmark turns the rates into the
//    special-function-unit ceiling of the forward kernel (one exponential per
//    score against 4 d tensor-core flops per score).
//  * The TMEM load with a max reduction that gives the forward kernel its row
//    maxima (tmem_ld128_max_wait), run on a caller tile so that a test can check
//    the maximum and the loaded values bit for bit.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/attn.h"
#include "ptx.cuh"

namespace {

using namespace attn;

constexpr int kDiagThreads = 512;  // four warps per SM sub-partition
constexpr int kDiagChains = 8;     // independent dependency chains per thread
constexpr int kDiagIters = 1024;

// Longest per-CTA duration (SM clock cycles) of each kernel, and a sink that
// keeps the results alive.
__device__ unsigned long long g_diag_cycles[2];
__device__ float g_diag_sink;

// Each thread runs kDiagChains chains x = ex2(-x): one special-function-unit
// instruction per step, no other arithmetic on the chain.
__global__ void __launch_bounds__(kDiagThreads, 1) diag_ex2_kernel(float seed) {
  float x[kDiagChains];
#pragma unroll
  for (int c = 0; c < kDiagChains; ++c) x[c] = seed + 0.01f * c + 1e-6f * threadIdx.x;
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < kDiagIters; ++it) {
#pragma unroll
    for (int c = 0; c < kDiagChains; ++c) x[c] = ex2_approx(-x[c]);
  }
  __syncthreads();
  const long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kDiagChains; ++c) s += x[c];
  if (s == 12345.f) g_diag_sink = s;
  if (threadIdx.x == 0) atomicMax(&g_diag_cycles[0], static_cast<unsigned long long>(t1 - t0));
}

// The same with the FMA-pipe exponential of the forward kernel, two scores per
// call: x = exp2_poly2(-x).
__global__ void __launch_bounds__(kDiagThreads, 1) diag_poly_kernel(float seed) {
  float2 x[kDiagChains / 2];
#pragma unroll
  for (int c = 0; c < kDiagChains / 2; ++c)
    x[c] = make_float2(seed + 0.01f * c + 1e-6f * threadIdx.x, seed - 0.01f * c);
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < kDiagIters; ++it) {
#pragma unroll
    for (int c = 0; c < kDiagChains / 2; ++c) x[c] = exp2_poly2(make_float2(-x[c].x, -x[c].y));
  }
  __syncthreads();
  const long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kDiagChains / 2; ++c) s += x[c].x + x[c].y;
  if (s == 12345.f) g_diag_sink = s;
  if (threadIdx.x == 0) atomicMax(&g_diag_cycles[1], static_cast<unsigned long long>(t1 - t0));
}

// y_poly[i] = exp2_poly2(x[i]), y_sfu[i] = ex2.approx.ftz(x[i]); the pairs of
// exp2_poly2 are (x[2i], x[2i+1]), a lone last element pairs with itself.
__global__ void diag_eval_kernel(const float* x, float* y_poly, float* y_sfu, long long n) {
  const long long pairs = (n + 1) / 2;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < pairs;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long a = 2 * i, b = 2 * i + 1 < n ? 2 * i + 1 : 2 * i;
    const float2 r = exp2_poly2(make_float2(x[a], x[b]));
    y_poly[a] = r.x;
    y_sfu[a] = ex2_approx(x[a]);
    if (b != a) {
      y_poly[b] = r.y;
      y_sfu[b] = ex2_approx(x[b]);
    }
  }
}

// One 128 x 128 f32 tile through TMEM: thread t writes row t of `in` into TMEM
// lane t, loads it back with tmem_ld128_max_wait and writes the values it got to
// `vals` and their maximum to `row_max[t]`; then with tmem_ld128_max32_wait, the
// maxima of its four groups of 32 columns to block_max[4 t ..] (if not null).
// 128 threads, one CTA; warp w reaches lanes 32 w .. 32 w + 31.
__global__ void __launch_bounds__(128, 1) diag_tmem_row_max_kernel(const float* in, float* vals, float* row_max,
                                                                   float* block_max) {
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x / 32;
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_slot), 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = tmem_slot + (static_cast<uint32_t>(32 * warp) << 16);
  const float* src = in + static_cast<size_t>(threadIdx.x) * 128;
#pragma unroll
  for (int c0 = 0; c0 < 128; c0 += 32) {
    uint32_t w[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) w[c] = __float_as_uint(src[c0 + c]);
    tmem_st32(taddr + c0, w);
  }
  tmem_st_wait();
  uint32_t r[128];
  float mx;
  tmem_ld128_max_wait(taddr, r, mx);
  float* dst = vals + static_cast<size_t>(threadIdx.x) * 128;
#pragma unroll
  for (int c = 0; c < 128; ++c) dst[c] = __uint_as_float(r[c]);
  row_max[threadIdx.x] = mx;
  if (block_max) {
    float bm[4];
    tmem_ld128_max32_wait(taddr, r, bm);
#pragma unroll
    for (int b = 0; b < 4; ++b) block_max[4 * threadIdx.x + b] = bm[b];
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem_slot, 128);
  }
}

}  // namespace

extern "C" int attn_diag_tmem_row_max(const float* in, float* vals, float* row_max, float* block_max,
                                      void* stream) {
  if (!in || !vals || !row_max) return ATTN_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(vals) | reinterpret_cast<uintptr_t>(row_max) |
       reinterpret_cast<uintptr_t>(block_max)) &
      3u)
    return ATTN_ERR_ALIGN;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (major != 10 || minor != 3) return ATTN_ERR_ARCH;
  diag_tmem_row_max_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(in, vals, row_max, block_max);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

extern "C" int attn_eval_exp2(const float* x, float* y_poly, float* y_sfu, long long n, void* stream) {
  if (!x || !y_poly || !y_sfu) return ATTN_ERR_NULL;
  if (n < 1) return ATTN_ERR_DIMS;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y_poly) | reinterpret_cast<uintptr_t>(y_sfu)) &
      3u)
    return ATTN_ERR_ALIGN;
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (major != 10 || minor != 3) return ATTN_ERR_ARCH;
  const long long pairs = (n + 1) / 2;
  long long blocks = (pairs + 255) / 256;
  if (blocks > 4ll * sms) blocks = 4ll * sms;
  diag_eval_kernel<<<static_cast<int>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(x, y_poly, y_sfu, n);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

extern "C" int attn_measure_exp2_rates(float* sfu_per_clk_sm, float* fma_poly_per_clk_sm, void* stream) {
  if (!sfu_per_clk_sm || !fma_poly_per_clk_sm) return ATTN_ERR_NULL;
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (major != 10 || minor != 3) return ATTN_ERR_ARCH;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const unsigned long long zero[2] = {0ull, 0ull};
  if (cudaMemcpyToSymbolAsync(g_diag_cycles, zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  // one untimed round of each (clocks and caches settle), then the measured one
  for (int rep = 0; rep < 2; ++rep) {
    if (rep == 1 &&
        cudaMemcpyToSymbolAsync(g_diag_cycles, zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return ATTN_ERR_CUDA;
    diag_ex2_kernel<<<sms, kDiagThreads, 0, s>>>(0.5f);
    diag_poly_kernel<<<sms, kDiagThreads, 0, s>>>(0.5f);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  }
  unsigned long long cyc[2] = {0ull, 0ull};
  if (cudaMemcpyFromSymbolAsync(cyc, g_diag_cycles, sizeof(cyc), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (cyc[0] == 0 || cyc[1] == 0) return ATTN_ERR_CUDA;
  const double per_cta = static_cast<double>(kDiagThreads) * kDiagChains * kDiagIters;
  *sfu_per_clk_sm = static_cast<float>(per_cta / static_cast<double>(cyc[0]));
  *fma_poly_per_clk_sm = static_cast<float>(per_cta / static_cast<double>(cyc[1]));
  return ATTN_OK;
}
