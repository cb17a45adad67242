// Gradients of exact attention on sm_103a: given Q, K, V, O, dO and the forward
// pass's per-row log-sum-exp, compute dQ, dK, dV without materialising P.
//
// Chain rule of o_i = sum_j p_ij v_j, p_i = softmax_j(scale q_i . k_j):
//   dV = P^T dO,  dP = dO V^T,  D_i = do_i . o_i,  dS = P o (dP - D),
//   dQ = scale dS K,  dK = scale dS^T Q.
// P is recomputed tile by tile from the stored log-sum-exp, p_ij =
// 2^(s_ij scale log2e - lse_i log2e), the same blockwise recomputation the forward
// pass uses instead of storing the N x N matrix (FlashAttention-2 article,
// "Background": tiling so the attention matrix is never materialised).
//
// Three kernels:
//   bwd_prep   D_i = do_i . o_i (one warp per row; memory-bound)
//   bwd_dq     unit = 128 query rows of one (b, h); loops over K/V blocks:
//              S = Q K^T and dP = dO V^T (SS MMAs), P and dS in registers,
//              dS (bf16) into TMEM, dQ += dS K (TS MMA, K read as an MN-major B)
//   bwd_dkdv   unit = 128 keys of one (b, h); loops over query blocks:
//              S^T = K Q^T and dP^T = V dO^T (SS MMAs), P^T and dS^T into TMEM,
//              dV += P^T dO and dK += dS^T Q (TS MMAs)
// Each CTA: warps 0-3 compute (thread t owns TMEM lane t = one row), warp 4 TMA
// producer, warp 5 single-thread MMA issuer (and TMEM owner).  dQ and dK/dV are
// separate passes, so no atomics are needed and the result is deterministic (two
// S-type products are computed twice).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "attn_fwd_kernel.cuh"  // tile layout, bounded waits, warp_wait
#include "ptx.cuh"

namespace attn {

constexpr int kBwdThreads = 192;
constexpr int kBwdProducerWarp = 4;
constexpr int kBwdMmaWarp = 5;

struct BwdParams {
  const __nv_bfloat16* o;     // [BH, N, D]   (prep)
  const __nv_bfloat16* dout;  // [BH, N, D]   (prep)
  const float* lse;           // [BH, N] natural-log row log-sum-exp of the forward pass
  float* dvec;                // [BH, N] D_i = do_i . o_i (workspace)
  __nv_bfloat16* dq;          // [BH, N, D]
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int BH, N;
  int num_blocks;             // ceil(N / 128)
  int num_units;              // BH * num_blocks
  int causal;
  float scale;
  float scale_log2;           // scale * log2(e)
  unsigned long long timeout_ns;
  int* err;
};

// ---------------------------------------------------------------------------
// D_i = sum_c do_ic o_ic in fp32; one warp per row, D/32 channels per lane.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const BwdParams p) {
  constexpr int kPer = D / 32;
  const int lane = threadIdx.x & 31;
  const long long rows = static_cast<long long>(p.BH) * p.N;
  const long long w0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long r = w0; r < rows; r += nw) {
    const __nv_bfloat16* a = p.o + r * D + lane * kPer;
    const __nv_bfloat16* b = p.dout + r * D + lane * kPer;
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < kPer; i += 2) {
      const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(a + i));
      const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(b + i));
      acc = fmaf(x.x, y.x, fmaf(x.y, y.y, acc));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) p.dvec[r] = acc;
  }
}

template <int D, int NS>
struct BwdSmem {
  using L = TileLayout<D, 2>;
  // two tiles loaded once per unit, then a ring of NS stages of two tiles
  static constexpr uint32_t kOnce = 0;
  static constexpr uint32_t kRing = 2 * L::kTileBytes;
  static constexpr uint32_t kExtra = kRing + 2 * NS * L::kTileBytes;  // lse/D vectors (dK/dV pass)
  static constexpr uint32_t kBars = kExtra + 2 * 2 * 128 * 4;
  static constexpr int kNumBars = 16 + 3 * NS;  // [9], [10]: vector barriers of the dK/dV pass
  static constexpr size_t kBytes = 1024 + kBars + 8 * kNumBars + 16;
  static_assert(kBytes <= 232448, "shared memory plan exceeds 227 KB");
};

// Bounded wait + abort plumbing shared by the two passes
#define ATTN_BWD_WAIT(bar, par, where) mbar_wait((bar), (par), abort_flag, tmo, p.err, (where))

// ---------------------------------------------------------------------------
// dQ pass.  TMEM: S at 0, dP at 128 (dS bf16 overwrites dP's first 64 columns),
// dQ accumulator at 256.
// ---------------------------------------------------------------------------
template <int D, int NS>
__global__ void __launch_bounds__(kBwdThreads, 1)
attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                   const BwdParams p) {
  using Sm = BwdSmem<D, NS>;
  using L = typename Sm::L;
  constexpr uint32_t kS = 0, kDP = 128, kDQ = 256;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const uint32_t sQ = base + Sm::kOnce, sDO = sQ + L::kTileBytes;
  const uint32_t sK = base + Sm::kRing, sV = sK + NS * L::kTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sm::kBars);
  const uint32_t b_qd_full = smem_u32(&bars[0]), b_qd_empty = smem_u32(&bars[1]);
  const uint32_t b_s_full = smem_u32(&bars[2]), b_s_free = smem_u32(&bars[3]);
  const uint32_t b_dp_full = smem_u32(&bars[4]), b_ds_ready = smem_u32(&bars[5]);
  const uint32_t b_dq_done = smem_u32(&bars[6]), b_dq_free = smem_u32(&bars[7]);
  const uint32_t b_drain = smem_u32(&bars[8]);
  const uint32_t b_k_full = smem_u32(&bars[16]), b_v_full = smem_u32(&bars[16 + NS]);
  const uint32_t b_kv_empty = smem_u32(&bars[16 + 2 * NS]);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bars[Sm::kNumBars]);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t tmo = p.timeout_ns;
  const int T = p.num_blocks;

  if (threadIdx.x == 0) {
    mbar_init(b_qd_full, 1);
    mbar_init(b_qd_empty, 1);
    mbar_init(b_s_full, 1);
    mbar_init(b_s_free, 128);
    mbar_init(b_dp_full, 1);
    mbar_init(b_ds_ready, 128);
    mbar_init(b_dq_done, 1);
    mbar_init(b_dq_free, 128);
    mbar_init(b_drain, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(b_k_full + 8 * s, 1);
      mbar_init(b_v_full + 8 * s, 1);
      mbar_init(b_kv_empty + 8 * s, 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kBwdMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // unit -> (bh, query block qb); causal: heaviest (last) query blocks first
  auto unit = [&](int u, int& bh, int& qb, int& nkv) {
    bh = u / T;
    const int r = u - bh * T;
    qb = p.causal ? (T - 1 - r) : r;
    nkv = p.causal ? qb + 1 : T;
  };
  auto unit_for_round = [&](int round) {
    const int G = gridDim.x, c = blockIdx.x;
    const int pos = round * G + ((round & 1) ? (G - 1 - c) : c);
    return pos < p.num_units ? pos : -1;
  };

  if (warp == kBwdProducerWarp) {
    if (lane == 0) {
      // Q and dO are read by this unit only; K and V by every query block of the head
      const uint64_t pol_once = l2_policy_evict_first(), pol_ring = l2_policy_evict_last();
      uint32_t g = 0;
      int units = 0;
      bool ok = true;
      for (int round = 0; ok; ++round) {
        const int u = unit_for_round(round);
        if (u < 0) break;
        int bh, qb, nkv;
        unit(u, bh, qb, nkv);
        if (units > 0 && !(ok = ATTN_BWD_WAIT(b_qd_empty, (units - 1) & 1, 40))) break;
        mbar_arrive_expect_tx(b_qd_full, 2 * L::kTileBytes);
        for (int c = 0; c < (int)L::kChunks; ++c) {
          tma_load_3d(sQ + c * L::kChunkBytes, &tmap_q, b_qd_full, c * 64, qb * kBlockM, bh, pol_once);
          tma_load_3d(sDO + c * L::kChunkBytes, &tmap_do, b_qd_full, c * 64, qb * kBlockM, bh, pol_once);
        }
        ++units;
        for (int j = 0; j < nkv; ++j, ++g) {
          const uint32_t st = g % NS, use = g / NS;
          if (use > 0 && !(ok = ATTN_BWD_WAIT(b_kv_empty + 8 * st, (use - 1) & 1, 41))) break;
          mbar_arrive_expect_tx(b_k_full + 8 * st, L::kTileBytes);
          for (int c = 0; c < (int)L::kChunks; ++c)
            tma_load_3d(sK + st * L::kTileBytes + c * L::kChunkBytes, &tmap_k, b_k_full + 8 * st, c * 64,
                        j * kBlockN, bh, pol_ring);
          mbar_arrive_expect_tx(b_v_full + 8 * st, L::kTileBytes);
          for (int c = 0; c < (int)L::kChunks; ++c)
            tma_load_3d(sV + st * L::kTileBytes + c * L::kChunkBytes, &tmap_v, b_v_full + 8 * st, c * 64,
                        j * kBlockN, bh, pol_ring);
        }
      }
      volatile int no_abort = 0;
      if (ok) {
        for (uint32_t i = (g > NS ? g - NS : 0); i < g; ++i)
          mbar_wait(b_kv_empty + 8 * (i % NS), (i / NS) & 1, abort_flag, tmo, p.err, 42);
        if (units > 0) mbar_wait(b_qd_empty, (units - 1) & 1, abort_flag, tmo, p.err, 43);
      } else {
        for (uint32_t i = (g > NS ? g - NS : 0); i < g; ++i) {
          mbar_wait(b_k_full + 8 * (i % NS), (i / NS) & 1, &no_abort, tmo, nullptr, 0);
          mbar_wait(b_v_full + 8 * (i % NS), (i / NS) & 1, &no_abort, tmo, nullptr, 0);
        }
        if (units > 0) mbar_wait(b_qd_full, (units - 1) & 1, &no_abort, tmo, nullptr, 0);
      }
    }
  } else if (warp == kBwdMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc_ss = make_idesc(kBlockM, kBlockN, 1, false);  // bf16, K-major A and B
      constexpr uint32_t idesc_dq = make_idesc(kBlockM, D, 1, true);        // B = K, MN-major
      // C (tmem) = A B^T with A, B 128 x D K-major tiles
      auto issue_ss = [&](uint32_t c_tmem, uint32_t a_base, uint32_t b_base) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kChunkBytes + (kk & 3) * 32;
          mma_f16_ss(c_tmem, sdesc_sw128(a_base + off, 16, 1024), sdesc_sw128(b_base + off, 16, 1024), idesc_ss,
                     kk > 0 ? 1u : 0u);
        }
      };
      uint32_t g = 0, s_iter = 0, ds_iter = 0;
      int units = 0;
      bool ok = true;
      for (int round = 0; ok; ++round) {
        const int u = unit_for_round(round);
        if (u < 0) break;
        int bh, qb, nkv;
        unit(u, bh, qb, nkv);
        if (!(ok = ATTN_BWD_WAIT(b_qd_full, units & 1, 50))) break;
        // S_0 and dP_0
        {
          const uint32_t st = g % NS, ph = (g / NS) & 1;
          if (!(ok = ATTN_BWD_WAIT(b_k_full + 8 * st, ph, 51))) break;
          if (s_iter > 0 && !(ok = ATTN_BWD_WAIT(b_s_free, (s_iter - 1) & 1, 52))) break;
          tc_fence_after();
          issue_ss(tmem + kS, sQ, sK + st * L::kTileBytes);
          mma_commit(b_s_full);
          ++s_iter;
          if (!(ok = ATTN_BWD_WAIT(b_v_full + 8 * st, ph, 53))) break;
          tc_fence_after();
          issue_ss(tmem + kDP, sDO, sV + st * L::kTileBytes);
          mma_commit(b_dp_full);
        }
        for (int j = 0; j < nkv && ok; ++j) {
          const uint32_t gj = g + j, st = gj % NS;
          const uint32_t stn = (gj + 1) % NS, phn = ((gj + 1) / NS) & 1;
          if (j + 1 < nkv) {
            // S_{j+1} may overwrite S once the compute warps have read S_j
            if (!(ok = ATTN_BWD_WAIT(b_k_full + 8 * stn, phn, 54))) break;
            if (!(ok = ATTN_BWD_WAIT(b_s_free, (s_iter - 1) & 1, 55))) break;
            tc_fence_after();
            issue_ss(tmem + kS, sQ, sK + stn * L::kTileBytes);
            mma_commit(b_s_full);
            ++s_iter;
          }
          if (!(ok = ATTN_BWD_WAIT(b_ds_ready, ds_iter & 1, 56))) break;
          ++ds_iter;
          if (j == 0 && units > 0 && !(ok = ATTN_BWD_WAIT(b_dq_free, (units - 1) & 1, 57))) break;
          tc_fence_after();
          // dQ += dS K_j: dS (bf16) in TMEM columns kDP..kDP+63, K_j as an MN-major B
#pragma unroll
          for (int kk = 0; kk < kBlockN / 16; ++kk)
            mma_f16_ts(tmem + kDQ, tmem + kDP + kk * 8,
                       sdesc_sw128(sK + st * L::kTileBytes + kk * 16 * 128, L::kChunkBytes, 1024), idesc_dq,
                       (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(b_kv_empty + 8 * st);
          if (j == nkv - 1) {
            mma_commit(b_dq_done);
            mma_commit(b_qd_empty);
          } else {
            // dP_{j+1} overwrites dS_j, which the dQ product above has consumed
            if (!(ok = ATTN_BWD_WAIT(b_v_full + 8 * stn, phn, 58))) break;
            tc_fence_after();
            issue_ss(tmem + kDP, sDO, sV + stn * L::kTileBytes);
            mma_commit(b_dp_full);
          }
        }
        g += nkv;
        ++units;
      }
      mma_commit(b_drain);
      volatile int no_abort = 0;
      mbar_wait(b_drain, 0, &no_abort, tmo, nullptr, 0);
    }
  } else {
    // ----------------------------------------------------------- compute
    const int t = threadIdx.x;  // query row within the tile = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float cs = p.scale_log2;
    uint32_t s_iter = 0, dp_iter = 0;
    int units = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const int u = unit_for_round(round);
      if (u < 0) break;
      int bh, qb, nkv;
      unit(u, bh, qb, nkv);
      const int row = qb * kBlockM + t;
      const bool valid = row < p.N;
      const size_t ridx = static_cast<size_t>(bh) * p.N + (valid ? row : 0);
      const float lse2 = valid ? __ldg(p.lse + ridx) * 1.4426950408889634f : 0.f;
      const float drow = valid ? __ldg(p.dvec + ridx) : 0.f;
      for (int j = 0; j < nkv; ++j) {
        if (!(ok = warp_wait(b_s_full, s_iter & 1, abort_flag, tmo, p.err, 60))) break;
        ++s_iter;
        tc_fence_after();
        uint32_t sraw[kBlockN];
        tmem_ld128_wait(tmem + lane_addr + kS, sraw);
        tc_fence_before();
        mbar_arrive(b_s_free);
        // P = 2^(s scale log2e - lse log2e); keys past N or past the row (causal) get 0
        const int key0 = j * kBlockN;
        int lim = p.N - 1 - key0;
        if (p.causal && row - key0 < lim) lim = row - key0;
        float pr[kBlockN];
#pragma unroll
        for (int c = 0; c < kBlockN; ++c) {
          const float e = ex2_approx(fmaf(__uint_as_float(sraw[c]), cs, -lse2));
          pr[c] = (valid && c <= lim) ? e : 0.f;
        }
        if (!(ok = warp_wait(b_dp_full, dp_iter & 1, abort_flag, tmo, p.err, 61))) break;
        ++dp_iter;
        tc_fence_after();
        // dS (scaled, bf16) into dP's first 64 columns for the dQ product; half h of
        // the keys is read from dP columns 64h.. before its dS lands in columns 32h..
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t dpr[64];
          tmem_ld64_wait(tmem + lane_addr + kDP + 64 * h, dpr);
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            const float d0 = pr[64 * h + c] * (__uint_as_float(dpr[c]) - drow) * p.scale;
            const float d1 = pr[64 * h + c + 1] * (__uint_as_float(dpr[c + 1]) - drow) * p.scale;
            pk[c / 2] = pack_bf16x2(d0, d1);
          }
          tmem_st32(tmem + lane_addr + kDP + 32 * h, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(b_ds_ready);
      }
      if (!ok) break;
      if (!(ok = warp_wait(b_dq_done, units & 1, abort_flag, tmo, p.err, 62))) break;
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < D / 64; ++h) {
        uint32_t o[64];
        tmem_ld64_wait(tmem + lane_addr + kDQ + 64 * h, o);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(p.dq + ridx * D + 64 * h);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_uint4(pack_bf16x2(__uint_as_float(o[8 * v]), __uint_as_float(o[8 * v + 1])),
                                pack_bf16x2(__uint_as_float(o[8 * v + 2]), __uint_as_float(o[8 * v + 3])),
                                pack_bf16x2(__uint_as_float(o[8 * v + 4]), __uint_as_float(o[8 * v + 5])),
                                pack_bf16x2(__uint_as_float(o[8 * v + 6]), __uint_as_float(o[8 * v + 7])));
        }
      }
      tc_fence_before();
      mbar_arrive(b_dq_free);
      ++units;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kBwdMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// dK / dV pass.  TMEM: S^T at 0 (P^T bf16 overwrites its first 64 columns),
// dP^T at 128 (dS^T bf16 overwrites its first 64 columns), dV at 256, dK at
// 256 + D.
// ---------------------------------------------------------------------------
template <int D, int NS>
__global__ void __launch_bounds__(kBwdThreads, 1)
attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                     const BwdParams p) {
  using Sm = BwdSmem<D, NS>;
  using L = typename Sm::L;
  constexpr uint32_t kS = 0, kDP = 128, kDV = 256, kDK = 256 + D;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const uint32_t sK = base + Sm::kOnce, sV = sK + L::kTileBytes;
  const uint32_t sQ = base + Sm::kRing, sDO = sQ + NS * L::kTileBytes;
  float* vec = reinterpret_cast<float*>(smem + Sm::kExtra);  // [2 buffers][lse2 | D][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sm::kBars);
  const uint32_t b_kv_full = smem_u32(&bars[0]), b_kv_empty = smem_u32(&bars[1]);
  const uint32_t b_st_full = smem_u32(&bars[2]), b_p_ready = smem_u32(&bars[3]);
  const uint32_t b_dpt_full = smem_u32(&bars[4]), b_ds_ready = smem_u32(&bars[5]);
  const uint32_t b_acc_done = smem_u32(&bars[6]), b_acc_free = smem_u32(&bars[7]);
  const uint32_t b_drain = smem_u32(&bars[8]);
  const uint32_t b_vec = smem_u32(&bars[9]);  // + 8 * buffer: the 128 vector values are in smem
  const uint32_t b_q_full = smem_u32(&bars[16]), b_do_full = smem_u32(&bars[16 + NS]);
  const uint32_t b_qdo_empty = smem_u32(&bars[16 + 2 * NS]);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bars[Sm::kNumBars]);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t tmo = p.timeout_ns;
  const int T = p.num_blocks;

  if (threadIdx.x == 0) {
    mbar_init(b_kv_full, 1);
    mbar_init(b_kv_empty, 1);
    mbar_init(b_st_full, 1);
    mbar_init(b_p_ready, 128);
    mbar_init(b_dpt_full, 1);
    mbar_init(b_ds_ready, 128);
    mbar_init(b_acc_done, 1);
    mbar_init(b_acc_free, 128);
    mbar_init(b_drain, 1);
    mbar_init(b_vec, 128);
    mbar_init(b_vec + 8, 128);
    for (int s = 0; s < NS; ++s) {
      mbar_init(b_q_full + 8 * s, 1);
      mbar_init(b_do_full + 8 * s, 1);
      mbar_init(b_qdo_empty + 8 * s, 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kBwdMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // unit -> (bh, key block kb); query blocks i0 .. T-1 (causal: i0 = kb, so the
  // first key blocks are the heaviest and run first)
  auto unit = [&](int u, int& bh, int& kb, int& i0) {
    bh = u / T;
    kb = u - bh * T;
    i0 = p.causal ? kb : 0;
  };
  auto unit_for_round = [&](int round) {
    const int G = gridDim.x, c = blockIdx.x;
    const int pos = round * G + ((round & 1) ? (G - 1 - c) : c);
    return pos < p.num_units ? pos : -1;
  };

  if (warp == kBwdProducerWarp) {
    if (lane == 0) {
      // K and V are read by this unit only; Q and dO by every key block of the head
      const uint64_t pol_once = l2_policy_evict_first(), pol_ring = l2_policy_evict_last();
      uint32_t g = 0;
      int units = 0;
      bool ok = true;
      for (int round = 0; ok; ++round) {
        const int u = unit_for_round(round);
        if (u < 0) break;
        int bh, kb, i0;
        unit(u, bh, kb, i0);
        if (units > 0 && !(ok = ATTN_BWD_WAIT(b_kv_empty, (units - 1) & 1, 70))) break;
        mbar_arrive_expect_tx(b_kv_full, 2 * L::kTileBytes);
        for (int c = 0; c < (int)L::kChunks; ++c) {
          tma_load_3d(sK + c * L::kChunkBytes, &tmap_k, b_kv_full, c * 64, kb * kBlockN, bh, pol_once);
          tma_load_3d(sV + c * L::kChunkBytes, &tmap_v, b_kv_full, c * 64, kb * kBlockN, bh, pol_once);
        }
        ++units;
        for (int i = i0; i < T; ++i, ++g) {
          const uint32_t st = g % NS, use = g / NS;
          if (use > 0 && !(ok = ATTN_BWD_WAIT(b_qdo_empty + 8 * st, (use - 1) & 1, 71))) break;
          mbar_arrive_expect_tx(b_q_full + 8 * st, L::kTileBytes);
          for (int c = 0; c < (int)L::kChunks; ++c)
            tma_load_3d(sQ + st * L::kTileBytes + c * L::kChunkBytes, &tmap_q, b_q_full + 8 * st, c * 64,
                        i * kBlockM, bh, pol_ring);
          mbar_arrive_expect_tx(b_do_full + 8 * st, L::kTileBytes);
          for (int c = 0; c < (int)L::kChunks; ++c)
            tma_load_3d(sDO + st * L::kTileBytes + c * L::kChunkBytes, &tmap_do, b_do_full + 8 * st, c * 64,
                        i * kBlockM, bh, pol_ring);
        }
      }
      volatile int no_abort = 0;
      if (ok) {
        for (uint32_t i = (g > NS ? g - NS : 0); i < g; ++i)
          mbar_wait(b_qdo_empty + 8 * (i % NS), (i / NS) & 1, abort_flag, tmo, p.err, 72);
        if (units > 0) mbar_wait(b_kv_empty, (units - 1) & 1, abort_flag, tmo, p.err, 73);
      } else {
        for (uint32_t i = (g > NS ? g - NS : 0); i < g; ++i) {
          mbar_wait(b_q_full + 8 * (i % NS), (i / NS) & 1, &no_abort, tmo, nullptr, 0);
          mbar_wait(b_do_full + 8 * (i % NS), (i / NS) & 1, &no_abort, tmo, nullptr, 0);
        }
        if (units > 0) mbar_wait(b_kv_full, (units - 1) & 1, &no_abort, tmo, nullptr, 0);
      }
    }
  } else if (warp == kBwdMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc_ss = make_idesc(kBlockM, kBlockN, 1, false);
      constexpr uint32_t idesc_acc = make_idesc(kBlockM, D, 1, true);  // B = dO or Q, MN-major
      auto issue_ss = [&](uint32_t c_tmem, uint32_t a_base, uint32_t b_base) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kChunkBytes + (kk & 3) * 32;
          mma_f16_ss(c_tmem, sdesc_sw128(a_base + off, 16, 1024), sdesc_sw128(b_base + off, 16, 1024), idesc_ss,
                     kk > 0 ? 1u : 0u);
        }
      };
      // acc (+)= A[tmem, 128 x 128 bf16 in 64 columns] B[smem, 128 rows x D, MN-major]
      auto issue_ts = [&](uint32_t acc_tmem, uint32_t a_tmem, uint32_t b_base, bool accumulate) {
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          mma_f16_ts(acc_tmem, a_tmem + kk * 8, sdesc_sw128(b_base + kk * 16 * 128, L::kChunkBytes, 1024),
                     idesc_acc, (accumulate || kk > 0) ? 1u : 0u);
      };
      uint32_t g = 0, p_iter = 0, ds_iter = 0;
      int units = 0;
      bool ok = true;
      for (int round = 0; ok; ++round) {
        const int u = unit_for_round(round);
        if (u < 0) break;
        int bh, kb, i0;
        unit(u, bh, kb, i0);
        const int n = T - i0;
        if (!(ok = ATTN_BWD_WAIT(b_kv_full, units & 1, 80))) break;
        {
          const uint32_t st = g % NS, ph = (g / NS) & 1;
          if (!(ok = ATTN_BWD_WAIT(b_q_full + 8 * st, ph, 81))) break;
          tc_fence_after();
          issue_ss(tmem + kS, sK, sQ + st * L::kTileBytes);   // S^T = K Q^T
          mma_commit(b_st_full);
          if (!(ok = ATTN_BWD_WAIT(b_do_full + 8 * st, ph, 82))) break;
          tc_fence_after();
          issue_ss(tmem + kDP, sV, sDO + st * L::kTileBytes);  // dP^T = V dO^T
          mma_commit(b_dpt_full);
        }
        for (int b = 0; b < n && ok; ++b) {
          const uint32_t gb = g + b, st = gb % NS;
          const uint32_t stn = (gb + 1) % NS, phn = ((gb + 1) / NS) & 1;
          // dV += P^T dO once the compute warps have written P^T
          if (!(ok = ATTN_BWD_WAIT(b_p_ready, p_iter & 1, 83))) break;
          ++p_iter;
          if (b == 0 && units > 0 && !(ok = ATTN_BWD_WAIT(b_acc_free, (units - 1) & 1, 84))) break;
          tc_fence_after();
          issue_ts(tmem + kDV, tmem + kS, sDO + st * L::kTileBytes, b > 0);
          if (b + 1 < n) {
            // S^T_{b+1} overwrites P^T_b, which the dV product above has consumed
            if (!(ok = ATTN_BWD_WAIT(b_q_full + 8 * stn, phn, 85))) break;
            tc_fence_after();
            issue_ss(tmem + kS, sK, sQ + stn * L::kTileBytes);
            mma_commit(b_st_full);
          }
          // dK += dS^T Q once the compute warps have written dS^T
          if (!(ok = ATTN_BWD_WAIT(b_ds_ready, ds_iter & 1, 86))) break;
          ++ds_iter;
          tc_fence_after();
          issue_ts(tmem + kDK, tmem + kDP, sQ + st * L::kTileBytes, b > 0);
          mma_commit(b_qdo_empty + 8 * st);
          if (b == n - 1) {
            mma_commit(b_acc_done);
            mma_commit(b_kv_empty);
          } else {
            if (!(ok = ATTN_BWD_WAIT(b_do_full + 8 * stn, phn, 87))) break;
            tc_fence_after();
            issue_ss(tmem + kDP, sV, sDO + stn * L::kTileBytes);
            mma_commit(b_dpt_full);
          }
        }
        g += n;
        ++units;
      }
      mma_commit(b_drain);
      volatile int no_abort = 0;
      mbar_wait(b_drain, 0, &no_abort, tmo, nullptr, 0);
    }
  } else {
    // ----------------------------------------------------------- compute
    const int t = threadIdx.x;  // key within the tile = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float cs = p.scale_log2;
    uint32_t st_iter = 0, dp_iter = 0, it = 0;
    int units = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const int u = unit_for_round(round);
      if (u < 0) break;
      int bh, kb, i0;
      unit(u, bh, kb, i0);
      const int key = kb * kBlockN + t;
      for (int i = i0; i < T; ++i, ++it) {
        // the block's 128 query log-sum-exps (log2 units) and D values, shared
        float* lse2v = vec + (it & 1) * 256;
        float* dv_ = lse2v + 128;
        {
          const int q = i * kBlockM + t;
          const size_t qi = static_cast<size_t>(bh) * p.N + q;
          lse2v[t] = q < p.N ? __ldg(p.lse + qi) * 1.4426950408889634f : INFINITY;
          dv_[t] = q < p.N ? __ldg(p.dvec + qi) : 0.f;
        }
        // every compute thread has stored its value before anyone reads the vectors;
        // a buffer is rewritten two blocks later, after all threads passed this point
        // for the block in between
        mbar_arrive(b_vec + 8 * (it & 1));
        if (!(ok = warp_wait(b_vec + 8 * (it & 1), (it >> 1) & 1, abort_flag, tmo, p.err, 93))) break;
        if (!(ok = warp_wait(b_st_full, st_iter & 1, abort_flag, tmo, p.err, 90))) break;
        ++st_iter;
        tc_fence_after();
        uint32_t sraw[kBlockM];
        tmem_ld128_wait(tmem + lane_addr + kS, sraw);
        // P^T[key][q] = 2^(s cs - lse2[q]); zero for queries before the key (causal)
        // and past N (lse2 = +inf)
        const int lim = (p.causal && i == kb) ? t : 0;  // first visible query in this block
        uint32_t pk[kBlockM / 2];  // P^T as bf16 pairs: the dV product's operand, reused for dS^T
#pragma unroll
        for (int c = 0; c < kBlockM; c += 2) {
          const float e0 = ex2_approx(fmaf(__uint_as_float(sraw[c]), cs, -lse2v[c]));
          const float e1 = ex2_approx(fmaf(__uint_as_float(sraw[c + 1]), cs, -lse2v[c + 1]));
          pk[c / 2] = pack_bf16x2(c >= lim ? e0 : 0.f, c + 1 >= lim ? e1 : 0.f);
        }
        tmem_st64(tmem + lane_addr + kS, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(b_p_ready);
        if (!(ok = warp_wait(b_dpt_full, dp_iter & 1, abort_flag, tmo, p.err, 91))) break;
        ++dp_iter;
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t dpr[64];
          tmem_ld64_wait(tmem + lane_addr + kDP + 64 * h, dpr);
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            const int q0 = 64 * h + c;
            const float2 pp = bf16x2_to_float2(pk[q0 / 2]);
            const float d0 = pp.x * (__uint_as_float(dpr[c]) - dv_[q0]) * p.scale;
            const float d1 = pp.y * (__uint_as_float(dpr[c + 1]) - dv_[q0 + 1]) * p.scale;
            pk[q0 / 2] = pack_bf16x2(d0, d1);
          }
        }
        tmem_st64(tmem + lane_addr + kDP, pk);  // dS^T (scaled) for the dK product
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(b_ds_ready);
      }
      if (!ok) break;
      if (!(ok = warp_wait(b_acc_done, units & 1, abort_flag, tmo, p.err, 92))) break;
      tc_fence_after();
      const bool valid = key < p.N;
      const size_t kidx = static_cast<size_t>(bh) * p.N + (valid ? key : 0);
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* outp = which == 0 ? p.dv : p.dk;
        const uint32_t col = which == 0 ? kDV : kDK;
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          uint32_t o[64];
          tmem_ld64_wait(tmem + lane_addr + col + 64 * h, o);
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(outp + kidx * D + 64 * h);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v] = make_uint4(pack_bf16x2(__uint_as_float(o[8 * v]), __uint_as_float(o[8 * v + 1])),
                                  pack_bf16x2(__uint_as_float(o[8 * v + 2]), __uint_as_float(o[8 * v + 3])),
                                  pack_bf16x2(__uint_as_float(o[8 * v + 4]), __uint_as_float(o[8 * v + 5])),
                                  pack_bf16x2(__uint_as_float(o[8 * v + 6]), __uint_as_float(o[8 * v + 7])));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(b_acc_free);
      ++units;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kBwdMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

#undef ATTN_BWD_WAIT

}  // namespace attn
