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
//   bwd_prep   per row: -lse log2e and -scale D_i into a padded workspace
//              (one warp per row; memory-bound)
//   bwd_dq     unit = 128 query rows of one (b, h); loops over K/V blocks:
//              S = Q K^T and dP = dO V^T (SS MMAs), P and dS in registers,
//              dS (bf16) into TMEM, dQ += dS K (TS MMA, K read as an MN-major B)
//   bwd_dkdv   unit = 128 keys of one (b, h); loops over query blocks:
//              S^T = K Q^T and dP^T = V dO^T (SS MMAs), P^T and dS^T into TMEM,
//              dV += P^T dO and dK += dS^T Q (TS MMAs)
// Each CTA of the dQ pass: warps 0-7 compute in two warpgroups -- thread t of
// warpgroup h owns TMEM lane t (one row of the tile) and columns 64h..64h+63 of
// each 128-column tile, and writes its bf16 result into the first 32 of those
// columns -- warp 8 is the TMA producer, warp 9 the MMA warp (one elected lane
// issues; TMEM owner).  The dK/dV pass does the same with four warpgroups of 32
// columns (warps 0-15), its producer and MMA warps 16 and 17.
// dQ and dK/dV are separate passes, so no atomics are needed and the result is
// deterministic (the two S-type products are computed in both passes).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "attn_fwd_kernel.cuh"  // tile layout, bounded waits, warp_wait
#include "ptx.cuh"

namespace attn {

constexpr int kBwdComputeThreads = 256;
constexpr int kBwdThreads = 320;
constexpr int kBwdProducerWarp = 8;
constexpr int kBwdMmaWarp = 9;
// The dK/dV pass: four compute warpgroups (a quarter of every tile's 128 columns
// each), then the TMA producer warp and the MMA warp.  Four warps per sub-partition
// overlap the recomputed softmax's chain of TMEM load, arithmetic and TMEM store,
// which bound the pass with two (same results bit for bit; the backward of B16 H16
// N4096 d64 +6.5%, of B1 H32 N16384 d128 causal +3.7%); the dQ pass gained nothing
// from four and keeps two.
constexpr int kDkdvWarpgroups = 4;
constexpr int kDkdvComputeThreads = 128 * kDkdvWarpgroups;
constexpr int kDkdvThreads = kDkdvComputeThreads + 64;
constexpr int kDkdvProducerWarp = kDkdvComputeThreads / 32;
constexpr int kDkdvMmaWarp = kDkdvProducerWarp + 1;

struct BwdParams {
  const __nv_bfloat16* o;     // [BH, N, D]   (prep)
  const __nv_bfloat16* dout;  // [BH, N, D]   (prep)
  const float* lse;           // [BH, N] natural-log row log-sum-exp of the forward pass (prep)
  float* nlse2;               // [BH, Npad] -lse_i log2(e); -inf for i >= N (workspace)
  float* nds;                 // [BH, Npad] -scale D_i; 0 for i >= N (workspace)
  __nv_bfloat16* dq;          // [BH, N, D]
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int BH, N, Npad;            // Npad = 128 * num_blocks
  int num_blocks;             // ceil(N / 128)
  int num_units;              // BH * num_blocks
  int order;                  // unit order: kBwdOrderHeads, kBwdOrderZigzag or kBwdOrderBlocks
  int causal;
  float scale;
  float scale_log2;           // scale * log2(e)
  unsigned long long timeout_ns;
  int* err;
};

// ---------------------------------------------------------------------------
// Per padded row r = (bh, i): D_i = sum_c do_ic o_ic in fp32, one warp per row.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const BwdParams p) {
  constexpr int kPer = D / 32;
  const int lane = threadIdx.x & 31;
  const long long rows = static_cast<long long>(p.BH) * p.Npad;
  const long long w0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long r = w0; r < rows; r += nw) {
    const long long bh = r / p.Npad;
    const int i = static_cast<int>(r - bh * p.Npad);
    float acc = 0.f, nl = -INFINITY;
    if (i < p.N) {
      const long long src = bh * p.N + i;
      const __nv_bfloat16* a = p.o + src * D + lane * kPer;
      const __nv_bfloat16* b = p.dout + src * D + lane * kPer;
#pragma unroll
      for (int c = 0; c < kPer; c += 2) {
        const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(a + c));
        const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(b + c));
        acc = fmaf(x.x, y.x, fmaf(x.y, y.y, acc));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      nl = -__ldg(p.lse + src) * 1.4426950408889634f;
    }
    if (lane == 0) {
      p.nlse2[r] = nl;
      p.nds[r] = -p.scale * acc;
    }
  }
}

// Shared memory of both passes: two tiles loaded once per unit, ring A (K in
// the dQ pass, Q in the dK/dV pass) of RA stages and ring B (V, dO) of RB
// stages.  Ring A's tile is read by the first and the last product of a step,
// ring B's only by the second, so ring B frees its stages sooner.
template <int D, int RA, int RB>
struct BwdSmem {
  using L = TileLayout<D, 2>;
  static constexpr uint32_t kOnce = 0;
  static constexpr uint32_t kRingA = 2 * L::kTileBytes;
  static constexpr uint32_t kRingB = kRingA + RA * L::kTileBytes;
  static constexpr uint32_t kBars = kRingB + RB * L::kTileBytes;
  static constexpr int kNumBars = 16 + 2 * (RA + RB);
  static constexpr size_t kBytes = 1024 + kBars + 8 * kNumBars + 16;
  static_assert(kBytes <= 232448, "shared memory plan exceeds 227 KB");
};

// acc (+)= A B with A = 128 x 128 bf16 in TMEM (two keys per column) laid out as
// kWG compute warpgroups write it: warpgroup w's 128 / kWG keys in the first half
// of its own 128 / kWG columns (two warpgroups: keys 0..63 in columns a_region +
// 0..31, keys 64..127 in a_region + 64..95); B = 128 rows x D at b_base, MN-major.
// (Descriptors as 32-bit low words: step kk adds its byte offset >> 4 to the
// address field, which never carries since shared memory stays below 2^18.)
template <typename L, int kWG = 2>
__device__ __forceinline__ void bwd_issue_ts(uint32_t acc, uint32_t a_region, uint32_t b_base, uint32_t idesc,
                                             bool accumulate) {
  const uint32_t b0 = sdesc_lo(b_base, L::kChunkBytes);
  constexpr uint32_t hi = sdesc_hi_sw128(1024);
  constexpr int kSteps = 8 / kWG;  // 16-key MMA steps per warpgroup
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_f16_ts_w(acc, a_region + (kk / kSteps) * (128 / kWG) + (kk % kSteps) * 8, b0 + ((kk * 16 * 128) >> 4),
                 hi, idesc, (accumulate || kk > 0) ? 1u : 0u);
}

// C = A B^T with A, B 128 x D K-major bf16 tiles.
template <int D, typename L>
__device__ __forceinline__ void bwd_issue_ss(uint32_t c_tmem, uint32_t a_base, uint32_t b_base, uint32_t idesc) {
  const uint32_t a0 = sdesc_lo(a_base, 16), b0 = sdesc_lo(b_base, 16);
  constexpr uint32_t hi = sdesc_hi_sw128(1024);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = ((kk >> 2) * L::kChunkBytes + (kk & 3) * 32) >> 4;
    mma_f16_ss_w(c_tmem, a0 + off, b0 + off, hi, idesc, kk > 0 ? 1u : 0u);
  }
}

// One thread's part of an accumulator row (kCols fp32 TMEM columns) -> bf16 at dst.
template <int kCols>
__device__ __forceinline__ void bwd_store_row_part(uint32_t taddr, __nv_bfloat16* dst, bool valid) {
  static_assert(kCols == 16 || kCols == 32 || kCols == 64, "16, 32 or 64 columns");
  uint32_t a[kCols];
  if constexpr (kCols == 64) {
    tmem_ld64_wait(taddr, a);
  } else if constexpr (kCols == 32) {
    tmem_ld32_wait(taddr, a);
  } else {
    tmem_ld16_wait(taddr, a);
  }
  if (valid) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int v = 0; v < kCols / 8; ++v)
      d4[v] = make_uint4(pack_bf16x2(__uint_as_float(a[8 * v]), __uint_as_float(a[8 * v + 1])),
                         pack_bf16x2(__uint_as_float(a[8 * v + 2]), __uint_as_float(a[8 * v + 3])),
                         pack_bf16x2(__uint_as_float(a[8 * v + 4]), __uint_as_float(a[8 * v + 5])),
                         pack_bf16x2(__uint_as_float(a[8 * v + 6]), __uint_as_float(a[8 * v + 7])));
  }
}

// The two load rings of a pass (mbarrier arrays, 8 bytes apart).
struct BwdRings {
  uint32_t a_full, a_empty, b_full, b_empty;
};

// Wait for what the producer issued to be consumed (ok) or to land (after an
// abort), so that no copy is in flight when the CTA exits.  ga / gb: tiles
// issued into ring A / B.
template <int RA, int RB>
__device__ __forceinline__ void bwd_producer_drain(bool ok, uint32_t ga, uint32_t gb, int units,
                                                   const BwdRings& rg, uint32_t once_full, uint32_t once_empty,
                                                   volatile int* abort_flag, uint64_t tmo, int* err, int where) {
  volatile int no_abort = 0;
  for (uint32_t i = (ga > RA ? ga - RA : 0); i < ga; ++i) {
    if (ok) mbar_wait(rg.a_empty + 8 * (i % RA), (i / RA) & 1, abort_flag, tmo, err, where);
    else mbar_wait(rg.a_full + 8 * (i % RA), (i / RA) & 1, &no_abort, tmo, nullptr, 0);
  }
  for (uint32_t i = (gb > RB ? gb - RB : 0); i < gb; ++i) {
    if (ok) mbar_wait(rg.b_empty + 8 * (i % RB), (i / RB) & 1, abort_flag, tmo, err, where);
    else mbar_wait(rg.b_full + 8 * (i % RB), (i / RB) & 1, &no_abort, tmo, nullptr, 0);
  }
  if (units > 0) {
    if (ok) mbar_wait(once_empty, (units - 1) & 1, abort_flag, tmo, err, where);
    else mbar_wait(once_full, (units - 1) & 1, &no_abort, tmo, nullptr, 0);
  }
}

// Unit order of both passes.  A unit is (bh, rank r) with r = 0 the heaviest block
// of a head under the causal mask (dq: the last query block; dkdv: the first key
// block); without the mask all blocks cost the same.
//   kBwdOrderHeads   head-major, heaviest first, dealt over the CTAs in a snake
//                    (mirror on odd rounds): the units of a head run together and
//                    share its streamed tensors in L2.
//   kBwdOrderZigzag  causal with at least four rounds of pairs: block pairs
//                    (r, T-1-r) of one head cost the same for every r; CTA k of a
//                    round takes pair k's heavy block in even iterations and its
//                    light one in odd iterations (an odd T leaves the middle block
//                    alone), head-major.
//   kBwdOrderBlocks  causal with fewer rounds and all heads' streamed tensors within
//                    L2: block-major, heaviest first over all heads, in the snake
//                    (~98% balance where head-major gives ~85%).
constexpr int kBwdOrderHeads = 0, kBwdOrderZigzag = 1, kBwdOrderBlocks = 2;
constexpr int kBwdDone = -1, kBwdSkip = -2;
struct BwdUnit {
  int status;  // 0, kBwdDone or kBwdSkip
  int bh, r;
};
__device__ __forceinline__ BwdUnit bwd_unit_for_round(int round, const BwdParams& p) {
  const int G = gridDim.x, c = blockIdx.x, T = p.num_blocks;
  BwdUnit u{0, 0, 0};
  if (p.order == kBwdOrderZigzag) {
    const int half = (T + 1) >> 1;
    const int k = (round >> 1) * G + c;
    if (k >= p.BH * half) {
      u.status = kBwdDone;
      return u;
    }
    u.bh = k / half;
    const int cc = k - u.bh * half;
    if ((round & 1) && T - 1 - cc == cc) {
      u.status = kBwdSkip;
      return u;
    }
    u.r = (round & 1) ? T - 1 - cc : cc;
    return u;
  }
  const int pos = round * G + ((round & 1) ? (G - 1 - c) : c);
  if (pos >= p.num_units) {
    u.status = kBwdDone;
    return u;
  }
  if (p.order == kBwdOrderBlocks) {
    u.r = pos / p.BH;
    u.bh = pos - u.r * p.BH;
  } else {
    u.bh = pos / T;
    u.r = pos - u.bh * T;
  }
  return u;
}

// Bounded wait + abort plumbing shared by the two passes
#define ATTN_BWD_WAIT(bar, par, where) mbar_wait((bar), (par), abort_flag, tmo, p.err, (where))
// the same, taken by a whole warp (same answer on every lane)
#define ATTN_BWD_WAIT_W(bar, par, where) warp_wait((bar), (par), abort_flag, tmo, p.err, (where))

// ---------------------------------------------------------------------------
// dQ pass.  TMEM: S at 0, dP at 128 (each warpgroup's dS, bf16, over the first
// half of its own dP columns), dQ accumulator at 256.
// ---------------------------------------------------------------------------
template <int D, int RA, int RB>
__global__ void __launch_bounds__(kBwdThreads, 1)
attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                   const BwdParams p) {
  using Sm = BwdSmem<D, RA, RB>;
  using L = typename Sm::L;
  constexpr uint32_t kS = 0, kDP = 128, kDQ = 256;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const uint32_t sQ = base + Sm::kOnce, sDO = sQ + L::kTileBytes;
  const uint32_t sK = base + Sm::kRingA, sV = base + Sm::kRingB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sm::kBars);
  const uint32_t b_qd_full = smem_u32(&bars[0]), b_qd_empty = smem_u32(&bars[1]);
  const uint32_t b_s_full = smem_u32(&bars[2]), b_s_free = smem_u32(&bars[3]);
  const uint32_t b_dp_full = smem_u32(&bars[4]), b_ds_ready = smem_u32(&bars[5]);
  const uint32_t b_dq_done = smem_u32(&bars[6]), b_dq_free = smem_u32(&bars[7]);
  const uint32_t b_drain = smem_u32(&bars[8]);
  const BwdRings rg{smem_u32(&bars[16]), smem_u32(&bars[16 + RA]), smem_u32(&bars[16 + 2 * RA]),
                    smem_u32(&bars[16 + 2 * RA + RB])};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bars[Sm::kNumBars]);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t tmo = p.timeout_ns;
  const int T = p.num_blocks;

  if (threadIdx.x == 0) {
    mbar_init(b_qd_full, 1);
    mbar_init(b_qd_empty, 1);
    mbar_init(b_s_full, 1);
    mbar_init(b_s_free, kBwdComputeThreads);
    mbar_init(b_dp_full, 1);
    mbar_init(b_ds_ready, kBwdComputeThreads);
    mbar_init(b_dq_done, 1);
    mbar_init(b_dq_free, kBwdComputeThreads);
    mbar_init(b_drain, 1);
    for (int s = 0; s < RA; ++s) {
      mbar_init(rg.a_full + 8 * s, 1);
      mbar_init(rg.a_empty + 8 * s, 1);
    }
    for (int s = 0; s < RB; ++s) {
      mbar_init(rg.b_full + 8 * s, 1);
      mbar_init(rg.b_empty + 8 * s, 1);
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
  auto unit = [&](const BwdUnit& uu, int& bh, int& qb, int& nkv) {
    bh = uu.bh;
    qb = p.causal ? (T - 1 - uu.r) : uu.r;
    nkv = p.causal ? qb + 1 : T;
  };

  if (warp == kBwdProducerWarp) {
    if (lane == 0) {
      // Q and dO are read by this unit only; K and V by every query block of the head
      const uint64_t pol_once = l2_policy_evict_first(), pol_ring = l2_policy_evict_last();
      uint32_t ga = 0, gb = 0;
      int units = 0;
      bool ok = true;
      for (int round = 0; ok; ++round) {
        const BwdUnit u = bwd_unit_for_round(round, p);
        if (u.status == kBwdDone) break;
        if (u.status == kBwdSkip) continue;
        int bh, qb, nkv;
        unit(u, bh, qb, nkv);
        if (units > 0 && !(ok = ATTN_BWD_WAIT(b_qd_empty, (units - 1) & 1, 40))) break;
        mbar_arrive_expect_tx(b_qd_full, 2 * L::kTileBytes);
        for (int c = 0; c < (int)L::kChunks; ++c) {
          tma_load_3d(sQ + c * L::kChunkBytes, &tmap_q, b_qd_full, c * 64, qb * kBlockM, bh, pol_once);
          tma_load_3d(sDO + c * L::kChunkBytes, &tmap_do, b_qd_full, c * 64, qb * kBlockM, bh, pol_once);
        }
        ++units;
        for (int j = 0; j < nkv; ++j) {
          const uint32_t sa = ga % RA, sb = gb % RB;
          if (ga >= RA && !(ok = ATTN_BWD_WAIT(rg.a_empty + 8 * sa, ((ga / RA) - 1) & 1, 41))) break;
          mbar_arrive_expect_tx(rg.a_full + 8 * sa, L::kTileBytes);
          for (int c = 0; c < (int)L::kChunks; ++c)
            tma_load_3d(sK + sa * L::kTileBytes + c * L::kChunkBytes, &tmap_k, rg.a_full + 8 * sa, c * 64,
                        j * kBlockN, bh, pol_ring);
          ++ga;
          if (gb >= RB && !(ok = ATTN_BWD_WAIT(rg.b_empty + 8 * sb, ((gb / RB) - 1) & 1, 42))) break;
          mbar_arrive_expect_tx(rg.b_full + 8 * sb, L::kTileBytes);
          for (int c = 0; c < (int)L::kChunks; ++c)
            tma_load_3d(sV + sb * L::kTileBytes + c * L::kChunkBytes, &tmap_v, rg.b_full + 8 * sb, c * 64,
                        j * kBlockN, bh, pol_ring);
          ++gb;
        }
      }
      bwd_producer_drain<RA, RB>(ok, ga, gb, units, rg, b_qd_full, b_qd_empty, abort_flag, tmo, p.err, 43);
    }
  } else if (warp == kBwdMmaWarp) {
    {  // whole warp, warp-uniform; one elected lane issues each MMA and commit
      constexpr uint32_t idesc_ss = make_idesc(kBlockM, kBlockN, 1, false);  // bf16, K-major A and B
      constexpr uint32_t idesc_dq = make_idesc(kBlockM, D, 1, true);        // B = K, MN-major
      uint32_t g = 0, s_iter = 0, ds_iter = 0;
      int units = 0;
      bool ok = true;
      for (int round = 0; ok; ++round) {
        const BwdUnit u = bwd_unit_for_round(round, p);
        if (u.status == kBwdDone) break;
        if (u.status == kBwdSkip) continue;
        int bh, qb, nkv;
        unit(u, bh, qb, nkv);
        if (!(ok = ATTN_BWD_WAIT_W(b_qd_full, units & 1, 50))) break;
        {  // S_0 and dP_0
          if (!(ok = ATTN_BWD_WAIT_W(rg.a_full + 8 * (g % RA), (g / RA) & 1, 51))) break;
          if (s_iter > 0 && !(ok = ATTN_BWD_WAIT_W(b_s_free, (s_iter - 1) & 1, 52))) break;
          tc_fence_after();
          bwd_issue_ss<D, L>(tmem + kS, sQ, sK + (g % RA) * L::kTileBytes, idesc_ss);
          mma_commit(b_s_full);
          ++s_iter;
          if (!(ok = ATTN_BWD_WAIT_W(rg.b_full + 8 * (g % RB), (g / RB) & 1, 53))) break;
          tc_fence_after();
          bwd_issue_ss<D, L>(tmem + kDP, sDO, sV + (g % RB) * L::kTileBytes, idesc_ss);
          mma_commit(b_dp_full);
          mma_commit(rg.b_empty + 8 * (g % RB));
          if (nkv == 1) mma_commit(b_qd_empty);  // Q and dO have no further reader
        }
        for (int j = 0; j < nkv && ok; ++j) {
          const uint32_t gj = g + j, gn = gj + 1;
          if (j + 1 < nkv) {
            // S_{j+1} may overwrite S once both warpgroups have read S_j
            if (!(ok = ATTN_BWD_WAIT_W(rg.a_full + 8 * (gn % RA), (gn / RA) & 1, 54))) break;
            if (!(ok = ATTN_BWD_WAIT_W(b_s_free, (s_iter - 1) & 1, 55))) break;
            tc_fence_after();
            bwd_issue_ss<D, L>(tmem + kS, sQ, sK + (gn % RA) * L::kTileBytes, idesc_ss);
            mma_commit(b_s_full);
            ++s_iter;
          }
          if (!(ok = ATTN_BWD_WAIT_W(b_ds_ready, ds_iter & 1, 56))) break;
          ++ds_iter;
          if (j == 0 && units > 0 && !(ok = ATTN_BWD_WAIT_W(b_dq_free, (units - 1) & 1, 57))) break;
          tc_fence_after();
          bwd_issue_ts<L>(tmem + kDQ, tmem + kDP, sK + (gj % RA) * L::kTileBytes, idesc_dq, j > 0);
          mma_commit(rg.a_empty + 8 * (gj % RA));
          if (j == nkv - 1) {
            mma_commit(b_dq_done);
          } else {
            // dP_{j+1} overwrites dS_j, which the dQ product above has consumed
            if (!(ok = ATTN_BWD_WAIT_W(rg.b_full + 8 * (gn % RB), (gn / RB) & 1, 58))) break;
            tc_fence_after();
            bwd_issue_ss<D, L>(tmem + kDP, sDO, sV + (gn % RB) * L::kTileBytes, idesc_ss);
            mma_commit(b_dp_full);
            mma_commit(rg.b_empty + 8 * (gn % RB));
            if (j + 2 == nkv) mma_commit(b_qd_empty);
          }
        }
        g += nkv;
        ++units;
      }
      mma_commit(b_drain);
      volatile int no_abort = 0;
      warp_wait(b_drain, 0, &no_abort, tmo, nullptr, 0);
    }
  } else {
    // ----------------------------------------------------------- compute
    const int wg = warp >> 2;         // column half of every tile
    const int t = threadIdx.x & 127;  // query row within the tile = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_addr + kS + 64 * wg, tP = tmem + lane_addr + kDP + 64 * wg;
    const float2 cs2 = make_float2(p.scale_log2, p.scale_log2);
    const float2 sc2 = make_float2(p.scale, p.scale);
    uint32_t s_iter = 0, dp_iter = 0;
    int units = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const BwdUnit u = bwd_unit_for_round(round, p);
      if (u.status == kBwdDone) break;
      if (u.status == kBwdSkip) continue;
      int bh, qb, nkv;
      unit(u, bh, qb, nkv);
      const int row = qb * kBlockM + t;
      const size_t vidx = static_cast<size_t>(bh) * p.Npad + row;
      const float nl = __ldg(p.nlse2 + vidx);  // -inf past N: P = 0 there
      const float2 nl2 = make_float2(nl, nl);
      const float nd = __ldg(p.nds + vidx);
      const float2 nd2 = make_float2(nd, nd);
      for (int j = 0; j < nkv; ++j) {
        if (!(ok = warp_wait(b_s_full, s_iter & 1, abort_flag, tmo, p.err, 60))) break;
        ++s_iter;
        tc_fence_after();
        uint32_t sraw[64];
        tmem_ld64_wait(tS, sraw);
        tc_fence_before();
        mbar_arrive(b_s_free);
        // P = 2^(s scale log2e - lse log2e); keys past N or past the row (causal) get 0
        float pr[64];
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float2 e = ffma2(make_float2(__uint_as_float(sraw[c]), __uint_as_float(sraw[c + 1])), cs2, nl2);
          pr[c] = ex2_approx(e.x);
          pr[c + 1] = ex2_approx(e.y);
        }
        const int key0 = j * kBlockN + 64 * wg;
        if ((p.causal && j == qb) || (j + 1) * kBlockN > p.N) {
          int lim = p.N - 1 - key0;
          if (p.causal && row - key0 < lim) lim = row - key0;
#pragma unroll
          for (int c = 0; c < 64; ++c) pr[c] = c <= lim ? pr[c] : 0.f;
        }
        if (!(ok = warp_wait(b_dp_full, dp_iter & 1, abort_flag, tmo, p.err, 61))) break;
        ++dp_iter;
        tc_fence_after();
        uint32_t dpr[64];
        tmem_ld64_wait(tP, dpr);
        // dS scale = P (scale dP - scale D), bf16, over the first half of this
        // warpgroup's dP columns (read in full above)
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float2 x = ffma2(make_float2(__uint_as_float(dpr[c]), __uint_as_float(dpr[c + 1])), sc2, nd2);
          const float2 ds = fmul2(x, make_float2(pr[c], pr[c + 1]));
          pk[c / 2] = pack_bf16x2(ds.x, ds.y);
        }
        tmem_st32(tP, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(b_ds_ready);
      }
      if (!ok) break;
      if (!(ok = warp_wait(b_dq_done, units & 1, abort_flag, tmo, p.err, 62))) break;
      tc_fence_after();
      const bool valid = row < p.N;
      bwd_store_row_part<D / 2>(tmem + lane_addr + kDQ + (D / 2) * wg,
                            p.dq + (static_cast<size_t>(bh) * p.N + (valid ? row : 0)) * D + (D / 2) * wg, valid);
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
// dK / dV pass.  TMEM: S^T at 0 (P^T, bf16, over the first half of each
// warpgroup's columns), dP^T at 128 (dS^T likewise), dV at 256, dK at 256 + D.
// ---------------------------------------------------------------------------
template <int D, int RA, int RB>
__global__ void __launch_bounds__(kDkdvThreads, 1)
attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                     const BwdParams p) {
  using Sm = BwdSmem<D, RA, RB>;
  using L = typename Sm::L;
  constexpr uint32_t kS = 0, kDP = 128, kDV = 256, kDK = 256 + D;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const uint32_t sK = base + Sm::kOnce, sV = sK + L::kTileBytes;
  const uint32_t sQ = base + Sm::kRingA, sDO = base + Sm::kRingB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sm::kBars);
  const uint32_t b_kv_full = smem_u32(&bars[0]), b_kv_empty = smem_u32(&bars[1]);
  const uint32_t b_st_full = smem_u32(&bars[2]), b_p_ready = smem_u32(&bars[3]);
  const uint32_t b_dpt_full = smem_u32(&bars[4]), b_ds_ready = smem_u32(&bars[5]);
  const uint32_t b_acc_done = smem_u32(&bars[6]), b_acc_free = smem_u32(&bars[7]);
  const uint32_t b_drain = smem_u32(&bars[8]);
  const BwdRings rg{smem_u32(&bars[16]), smem_u32(&bars[16 + RA]), smem_u32(&bars[16 + 2 * RA]),
                    smem_u32(&bars[16 + 2 * RA + RB])};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bars[Sm::kNumBars]);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t tmo = p.timeout_ns;
  const int T = p.num_blocks;

  if (threadIdx.x == 0) {
    mbar_init(b_kv_full, 1);
    mbar_init(b_kv_empty, 1);
    mbar_init(b_st_full, 1);
    mbar_init(b_p_ready, kDkdvComputeThreads);
    mbar_init(b_dpt_full, 1);
    mbar_init(b_ds_ready, kDkdvComputeThreads);
    mbar_init(b_acc_done, 1);
    mbar_init(b_acc_free, kDkdvComputeThreads);
    mbar_init(b_drain, 1);
    for (int s = 0; s < RA; ++s) {
      mbar_init(rg.a_full + 8 * s, 1);
      mbar_init(rg.a_empty + 8 * s, 1);
    }
    for (int s = 0; s < RB; ++s) {
      mbar_init(rg.b_full + 8 * s, 1);
      mbar_init(rg.b_empty + 8 * s, 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kDkdvMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // unit -> (bh, key block kb); query blocks i0 .. T-1 (causal: i0 = kb, so the
  // first key blocks are the heaviest and run first)
  auto unit = [&](const BwdUnit& uu, int& bh, int& kb, int& i0) {
    bh = uu.bh;
    kb = uu.r;
    i0 = p.causal ? kb : 0;
  };

  if (warp == kDkdvProducerWarp) {
    if (lane == 0) {
      // K and V are read by this unit only; Q and dO by every key block of the head
      const uint64_t pol_once = l2_policy_evict_first(), pol_ring = l2_policy_evict_last();
      uint32_t ga = 0, gb = 0;
      int units = 0;
      bool ok = true;
      for (int round = 0; ok; ++round) {
        const BwdUnit u = bwd_unit_for_round(round, p);
        if (u.status == kBwdDone) break;
        if (u.status == kBwdSkip) continue;
        int bh, kb, i0;
        unit(u, bh, kb, i0);
        if (units > 0 && !(ok = ATTN_BWD_WAIT(b_kv_empty, (units - 1) & 1, 70))) break;
        mbar_arrive_expect_tx(b_kv_full, 2 * L::kTileBytes);
        for (int c = 0; c < (int)L::kChunks; ++c) {
          tma_load_3d(sK + c * L::kChunkBytes, &tmap_k, b_kv_full, c * 64, kb * kBlockN, bh, pol_once);
          tma_load_3d(sV + c * L::kChunkBytes, &tmap_v, b_kv_full, c * 64, kb * kBlockN, bh, pol_once);
        }
        ++units;
        for (int i = i0; i < T; ++i) {
          const uint32_t sa = ga % RA, sb = gb % RB;
          if (ga >= RA && !(ok = ATTN_BWD_WAIT(rg.a_empty + 8 * sa, ((ga / RA) - 1) & 1, 71))) break;
          mbar_arrive_expect_tx(rg.a_full + 8 * sa, L::kTileBytes);
          for (int c = 0; c < (int)L::kChunks; ++c)
            tma_load_3d(sQ + sa * L::kTileBytes + c * L::kChunkBytes, &tmap_q, rg.a_full + 8 * sa, c * 64,
                        i * kBlockM, bh, pol_ring);
          ++ga;
          if (gb >= RB && !(ok = ATTN_BWD_WAIT(rg.b_empty + 8 * sb, ((gb / RB) - 1) & 1, 72))) break;
          mbar_arrive_expect_tx(rg.b_full + 8 * sb, L::kTileBytes);
          for (int c = 0; c < (int)L::kChunks; ++c)
            tma_load_3d(sDO + sb * L::kTileBytes + c * L::kChunkBytes, &tmap_do, rg.b_full + 8 * sb, c * 64,
                        i * kBlockM, bh, pol_ring);
          ++gb;
        }
      }
      bwd_producer_drain<RA, RB>(ok, ga, gb, units, rg, b_kv_full, b_kv_empty, abort_flag, tmo, p.err, 73);
    }
  } else if (warp == kDkdvMmaWarp) {
    {  // whole warp, warp-uniform; one elected lane issues each MMA and commit
      constexpr uint32_t idesc_ss = make_idesc(kBlockM, kBlockN, 1, false);
      constexpr uint32_t idesc_acc = make_idesc(kBlockM, D, 1, true);  // B = dO or Q, MN-major
      uint32_t g = 0, p_iter = 0, ds_iter = 0;
      int units = 0;
      bool ok = true;
      for (int round = 0; ok; ++round) {
        const BwdUnit u = bwd_unit_for_round(round, p);
        if (u.status == kBwdDone) break;
        if (u.status == kBwdSkip) continue;
        int bh, kb, i0;
        unit(u, bh, kb, i0);
        const int n = T - i0;
        if (!(ok = ATTN_BWD_WAIT_W(b_kv_full, units & 1, 80))) break;
        {  // S^T_0 = K Q_0^T and dP^T_0 = V dO_0^T
          if (!(ok = ATTN_BWD_WAIT_W(rg.a_full + 8 * (g % RA), (g / RA) & 1, 81))) break;
          tc_fence_after();
          bwd_issue_ss<D, L>(tmem + kS, sK, sQ + (g % RA) * L::kTileBytes, idesc_ss);
          mma_commit(b_st_full);
          if (!(ok = ATTN_BWD_WAIT_W(rg.b_full + 8 * (g % RB), (g / RB) & 1, 82))) break;
          tc_fence_after();
          bwd_issue_ss<D, L>(tmem + kDP, sV, sDO + (g % RB) * L::kTileBytes, idesc_ss);
          mma_commit(b_dpt_full);
          if (n == 1) mma_commit(b_kv_empty);  // K and V have no further reader
        }
        for (int b = 0; b < n && ok; ++b) {
          const uint32_t gb = g + b, gn = gb + 1;
          // dV += P^T dO once both warpgroups have written P^T
          if (!(ok = ATTN_BWD_WAIT_W(b_p_ready, p_iter & 1, 83))) break;
          ++p_iter;
          if (b == 0 && units > 0 && !(ok = ATTN_BWD_WAIT_W(b_acc_free, (units - 1) & 1, 84))) break;
          tc_fence_after();
          bwd_issue_ts<L, kDkdvWarpgroups>(tmem + kDV, tmem + kS, sDO + (gb % RB) * L::kTileBytes, idesc_acc, b > 0);
          mma_commit(rg.b_empty + 8 * (gb % RB));
          if (b + 1 < n) {
            // S^T_{b+1} overwrites P^T_b, which the dV product above has consumed
            if (!(ok = ATTN_BWD_WAIT_W(rg.a_full + 8 * (gn % RA), (gn / RA) & 1, 85))) break;
            tc_fence_after();
            bwd_issue_ss<D, L>(tmem + kS, sK, sQ + (gn % RA) * L::kTileBytes, idesc_ss);
            mma_commit(b_st_full);
          }
          // dK += dS^T Q once both warpgroups have written dS^T
          if (!(ok = ATTN_BWD_WAIT_W(b_ds_ready, ds_iter & 1, 86))) break;
          ++ds_iter;
          tc_fence_after();
          bwd_issue_ts<L, kDkdvWarpgroups>(tmem + kDK, tmem + kDP, sQ + (gb % RA) * L::kTileBytes, idesc_acc, b > 0);
          mma_commit(rg.a_empty + 8 * (gb % RA));
          if (b == n - 1) {
            mma_commit(b_acc_done);
          } else {
            // dP^T_{b+1} overwrites dS^T_b, which the dK product above has consumed
            if (!(ok = ATTN_BWD_WAIT_W(rg.b_full + 8 * (gn % RB), (gn / RB) & 1, 87))) break;
            tc_fence_after();
            bwd_issue_ss<D, L>(tmem + kDP, sV, sDO + (gn % RB) * L::kTileBytes, idesc_ss);
            mma_commit(b_dpt_full);
            if (b + 2 == n) mma_commit(b_kv_empty);
          }
        }
        g += n;
        ++units;
      }
      mma_commit(b_drain);
      volatile int no_abort = 0;
      warp_wait(b_drain, 0, &no_abort, tmo, nullptr, 0);
    }
  } else {
    // ----------------------------------------------------------- compute
    constexpr int kQ = kBlockM / kDkdvWarpgroups;  // this warpgroup's queries (columns) of a tile
    const int wg = warp >> 2;         // column quarter of every tile
    const int t = threadIdx.x & 127;  // key within the tile = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_addr + kS + kQ * wg, tP = tmem + lane_addr + kDP + kQ * wg;
    const float2 cs2 = make_float2(p.scale_log2, p.scale_log2);
    const float2 sc2 = make_float2(p.scale, p.scale);
    uint32_t st_iter = 0, dp_iter = 0;
    int units = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const BwdUnit u = bwd_unit_for_round(round, p);
      if (u.status == kBwdDone) break;
      if (u.status == kBwdSkip) continue;
      int bh, kb, i0;
      unit(u, bh, kb, i0);
      const int key = kb * kBlockN + t;
      for (int i = i0; i < T; ++i) {
        // this warpgroup's kQ queries of block i: -lse log2e and -scale D, from
        // the padded workspace (16-byte aligned; -inf and 0 past N)
        const size_t voff = static_cast<size_t>(bh) * p.Npad + i * kBlockM + kQ * wg;
        const float4* nl4 = reinterpret_cast<const float4*>(p.nlse2 + voff);
        const float4* nd4 = reinterpret_cast<const float4*>(p.nds + voff);
        float4 nl[kQ / 4];
#pragma unroll
        for (int c = 0; c < kQ / 4; ++c) nl[c] = __ldg(nl4 + c);
        if (!(ok = warp_wait(b_st_full, st_iter & 1, abort_flag, tmo, p.err, 90))) break;
        ++st_iter;
        tc_fence_after();
        uint32_t sraw[kQ];
        tmem_ld32_wait(tS, sraw);
        // P^T[key][q] = 2^(s scale log2e - lse_q log2e); zero for queries before
        // the key (causal diagonal block) and past N (lse = +inf)
        uint32_t pk[kQ / 2];
#pragma unroll
        for (int c = 0; c < kQ; c += 4) {
          const float4 l = nl[c / 4];
          const float2 e0 = ffma2(make_float2(__uint_as_float(sraw[c]), __uint_as_float(sraw[c + 1])), cs2,
                                  make_float2(l.x, l.y));
          const float2 e1 = ffma2(make_float2(__uint_as_float(sraw[c + 2]), __uint_as_float(sraw[c + 3])), cs2,
                                  make_float2(l.z, l.w));
          pk[c / 2] = pack_bf16x2(ex2_approx(e0.x), ex2_approx(e0.y));
          pk[c / 2 + 1] = pack_bf16x2(ex2_approx(e1.x), ex2_approx(e1.y));
        }
        if (p.causal && i == kb) {
          // query kQ wg + c is visible to key t iff kQ wg + c >= t
          const int first = t - kQ * wg;
#pragma unroll
          for (int c = 0; c < kQ; c += 2) {
            const uint32_t lo = c >= first ? 0x0000ffffu : 0u, hi = c + 1 >= first ? 0xffff0000u : 0u;
            pk[c / 2] &= lo | hi;
          }
        }
        tmem_st16(tS, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(b_p_ready);
        float4 nd[kQ / 4];
#pragma unroll
        for (int c = 0; c < kQ / 4; ++c) nd[c] = __ldg(nd4 + c);
        if (!(ok = warp_wait(b_dpt_full, dp_iter & 1, abort_flag, tmo, p.err, 91))) break;
        ++dp_iter;
        tc_fence_after();
        uint32_t dpr[kQ];
        tmem_ld32_wait(tP, dpr);
        // dS^T scale = P^T (scale dP^T - scale D), from the bf16 P^T of the dV product
#pragma unroll
        for (int c = 0; c < kQ; c += 4) {
          const float4 d = nd[c / 4];
          const float2 x0 = ffma2(make_float2(__uint_as_float(dpr[c]), __uint_as_float(dpr[c + 1])), sc2,
                                  make_float2(d.x, d.y));
          const float2 x1 = ffma2(make_float2(__uint_as_float(dpr[c + 2]), __uint_as_float(dpr[c + 3])), sc2,
                                  make_float2(d.z, d.w));
          const float2 ds0 = fmul2(x0, bf16x2_to_float2(pk[c / 2]));
          const float2 ds1 = fmul2(x1, bf16x2_to_float2(pk[c / 2 + 1]));
          pk[c / 2] = pack_bf16x2(ds0.x, ds0.y);
          pk[c / 2 + 1] = pack_bf16x2(ds1.x, ds1.y);
        }
        tmem_st16(tP, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(b_ds_ready);
      }
      if (!ok) break;
      if (!(ok = warp_wait(b_acc_done, units & 1, abort_flag, tmo, p.err, 92))) break;
      tc_fence_after();
      const bool valid = key < p.N;
      constexpr int kC = D / kDkdvWarpgroups;  // this warpgroup's columns of dK and dV
      const size_t kidx = (static_cast<size_t>(bh) * p.N + (valid ? key : 0)) * D + kC * wg;
      bwd_store_row_part<kC>(tmem + lane_addr + kDV + kC * wg, p.dv + kidx, valid);
      bwd_store_row_part<kC>(tmem + lane_addr + kDK + kC * wg, p.dk + kidx, valid);
      tc_fence_before();
      mbar_arrive(b_acc_free);
      ++units;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kDkdvMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

#undef ATTN_BWD_WAIT

}  // namespace attn
