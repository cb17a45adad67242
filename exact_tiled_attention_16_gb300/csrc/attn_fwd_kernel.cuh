// Exact attention forward pass on sm_103a: O = softmax(scale * Q K^T [+ causal mask]) V
// and the per-row log-sum-exp, computed tile by tile with the online softmax so
// that the N x N score matrix never leaves the SM.
//
// Method (FlashAttention-2 article, "Technical architecture": fewer non-matmul
// operations, parallelism over the sequence, work split inside a block; news
// article "FlashAttention scaling ..." section 1: rescaling deferred to the end of
// the inner loop, outer loop over Q blocks and inner loop over K/V blocks, a
// dedicated copy engine (TMA) and producer/consumer warp roles; ring-attention
// page, "technical insight": running max and running normaliser with earlier
// partial sums rescaled when a larger score arrives).
//
// Blackwell mapping of those ideas, one CTA per SM (persistent):
//   warps 0-3  softmax: thread t owns query row t of the 128-row tile (TMEM lane t)
//   warp  4    producer: TMA loads of Q once per tile and of K/V blocks into a
//              ring of NSTAGE shared-memory stages
//   warp  5    MMA issuer: S = Q K^T into TMEM (double-buffered), O += P V with P
//              read from TMEM; also owns the TMEM allocation
// TMEM columns: S buffers at 0 and 128 (fp32), O at 256 (D fp32 columns),
// P at 384 (128 keys as bf16 pairs = 64 columns).
//
// Work unit = (b*H + h, 128-row query block).  Units are handed out statically:
// unit u of the run order goes to CTA (u mod G) on even rounds and to the mirror
// CTA on odd rounds, so heavy and light causal units interleave across CTAs.
// The run order is head-major so that concurrently running units share K/V in L2,
// and under the causal mask each head's query blocks run from the heaviest (last)
// to the lightest.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace attn {

constexpr int kBlockM = 128;     // query rows per tile (= TMEM lanes)
constexpr int kBlockN = 128;     // keys per K/V block
constexpr int kNumThreads = 192; // 6 warps
constexpr int kSoftmaxWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS0 = 0, kTmemS1 = 128, kTmemO = 256, kTmemP = 384;
// The running max is only moved when a block raises it by more than this many
// powers of two; until then exponentials are taken against the stale max and are
// at most 2^kRescaleThreshold, which bf16 P and the fp32 accumulators absorb.
constexpr float kRescaleThreshold = 8.0f;

struct FwdParams {
  __nv_bfloat16* o;   // [B*H, N, D]
  float* lse;         // [B*H, N] or nullptr
  int BH;             // B*H
  int N;
  int num_qblocks;    // ceil(N / 128)
  int num_units;      // BH * num_qblocks
  int causal;
  float scale_log2;   // scale * log2(e)
  unsigned long long timeout_ns;
  int* err;           // device error word (first failure wins)
};

template <int D>
struct SmemLayout {
  static constexpr uint32_t kChunkBytes = kBlockM * 128;            // 128 rows x 128 bytes
  static constexpr uint32_t kChunks = D / 64;                       // 64 bf16 per 128-byte row
  static constexpr uint32_t kTileBytes = kChunks * kChunkBytes;     // one 128 x D bf16 tile
};

__device__ __forceinline__ void unit_coords(int u, int num_qblocks, int causal, int& bh, int& qb) {
  bh = u / num_qblocks;
  const int r = u - bh * num_qblocks;
  qb = causal ? (num_qblocks - 1 - r) : r;
}

// The unit index processed by this CTA in its `round`-th iteration (or -1).
__device__ __forceinline__ int unit_for_round(int round, int num_units) {
  const int G = gridDim.x;
  const int c = blockIdx.x;
  const int pos = round * G + ((round & 1) ? (G - 1 - c) : c);
  return pos < num_units ? pos : -1;
}

__device__ __forceinline__ int num_kv_blocks(int qb, int N, int causal) {
  const int all = (N + kBlockN - 1) / kBlockN;
  if (!causal) return all;
  const int lim = qb + 1;  // kBlockM == kBlockN: keys up to the tile's last row
  return lim < all ? lim : all;
}

// A wait taken by all 32 lanes of a warp that returns the same answer on every
// lane, so that the warp stays converged for the .sync.aligned tcgen05 ops.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t timeout_ns, int* err_word, int where) {
  const bool ok = mbar_wait(bar, parity, abort_flag, timeout_ns, err_word, where);
  return __all_sync(0xffffffffu, ok);
}

template <int D, int NSTAGE>
__global__ void __launch_bounds__(kNumThreads, 1)
attn_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const FwdParams p) {
  using L = SmemLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle atoms.
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);

  const uint32_t sQ = base;
  const uint32_t sK = sQ + L::kTileBytes;
  const uint32_t sV = sK + NSTAGE * L::kTileBytes;
  uint8_t* ctrl = smem + L::kTileBytes * (1 + 2 * NSTAGE);
  // barriers (8 bytes each)
  uint64_t* bars = reinterpret_cast<uint64_t*>(ctrl);
  const uint32_t b_q_full = smem_u32(&bars[0]);
  const uint32_t b_q_empty = smem_u32(&bars[1]);
  const uint32_t b_pv_done = smem_u32(&bars[2]);
  const uint32_t b_p_full = smem_u32(&bars[3]);
  const uint32_t b_o_free = smem_u32(&bars[4]);
  const uint32_t b_s_full0 = smem_u32(&bars[5]);   // +8*b for buffer b
  const uint32_t b_s_free0 = smem_u32(&bars[7]);
  const uint32_t b_drain = smem_u32(&bars[9]);
  const uint32_t b_k_full0 = smem_u32(&bars[10]);  // +8*stage
  const uint32_t b_v_full0 = smem_u32(&bars[10 + NSTAGE]);
  const uint32_t b_kv_empty0 = smem_u32(&bars[10 + 2 * NSTAGE]);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 8 * (10 + 3 * NSTAGE));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t tmo = p.timeout_ns;

  if (threadIdx.x == 0) {
    mbar_init(b_q_full, 1);
    mbar_init(b_q_empty, 1);
    mbar_init(b_pv_done, 1);
    mbar_init(b_p_full, kSoftmaxWarps * 32);
    mbar_init(b_o_free, kSoftmaxWarps * 32);
    mbar_init(b_s_full0, 1);
    mbar_init(b_s_full0 + 8, 1);
    mbar_init(b_s_free0, kSoftmaxWarps * 32);
    mbar_init(b_s_free0 + 8, kSoftmaxWarps * 32);
    mbar_init(b_drain, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(b_k_full0 + 8 * s, 1);
      mbar_init(b_v_full0 + 8 * s, 1);
      mbar_init(b_kv_empty0 + 8 * s, 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ TMA
    if (lane == 0) {
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      uint32_t kv_iter = 0;
      int tiles = 0;
      bool ok = true;
      for (int round = 0; ok; ++round) {
        const int u = unit_for_round(round, p.num_units);
        if (u < 0) break;
        int bh, qb;
        unit_coords(u, p.num_qblocks, p.causal, bh, qb);
        const int nkv = num_kv_blocks(qb, p.N, p.causal);
        if (tiles > 0 && !(ok = mbar_wait(b_q_empty, (tiles - 1) & 1, abort_flag, tmo, p.err, 1))) break;
        mbar_arrive_expect_tx(b_q_full, L::kTileBytes);
        for (int c = 0; c < (int)L::kChunks; ++c)
          tma_load_3d(sQ + c * L::kChunkBytes, &tmap_q, b_q_full, c * 64, qb * kBlockM, bh, pol_q);
        for (int j = 0; j < nkv; ++j, ++kv_iter) {
          const uint32_t st = kv_iter % NSTAGE;
          const uint32_t use = kv_iter / NSTAGE;
          if (use > 0 && !(ok = mbar_wait(b_kv_empty0 + 8 * st, (use - 1) & 1, abort_flag, tmo, p.err, 2)))
            break;
          mbar_arrive_expect_tx(b_k_full0 + 8 * st, L::kTileBytes);
          for (int c = 0; c < (int)L::kChunks; ++c)
            tma_load_3d(sK + st * L::kTileBytes + c * L::kChunkBytes, &tmap_k, b_k_full0 + 8 * st, c * 64,
                        j * kBlockN, bh, pol_kv);
          mbar_arrive_expect_tx(b_v_full0 + 8 * st, L::kTileBytes);
          for (int c = 0; c < (int)L::kChunks; ++c)
            tma_load_3d(sV + st * L::kTileBytes + c * L::kChunkBytes, &tmap_v, b_v_full0 + 8 * st, c * 64,
                        j * kBlockN, bh, pol_kv);
        }
        ++tiles;
      }
      // Tail: every copy issued has landed and every MMA commit that frees a
      // stage has arrived before the CTA may exit.  Waits are bounded.
      if (ok) {
        for (uint32_t i = (kv_iter > NSTAGE ? kv_iter - NSTAGE : 0); i < kv_iter; ++i) {
          const uint32_t st = i % NSTAGE, use = i / NSTAGE;
          mbar_wait(b_kv_empty0 + 8 * st, use & 1, abort_flag, tmo, p.err, 3);
        }
        if (tiles > 0) mbar_wait(b_q_empty, (tiles - 1) & 1, abort_flag, tmo, p.err, 4);
      } else {
        // Error path: wait (bounded, ignoring the abort flag) for our own copies.
        volatile int no_abort = 0;
        for (uint32_t i = (kv_iter > NSTAGE ? kv_iter - NSTAGE : 0); i < kv_iter; ++i) {
          const uint32_t st = i % NSTAGE, use = i / NSTAGE;
          mbar_wait(b_k_full0 + 8 * st, use & 1, &no_abort, tmo, nullptr, 0);
          mbar_wait(b_v_full0 + 8 * st, use & 1, &no_abort, tmo, nullptr, 0);
        }
        if (tiles > 0) mbar_wait(b_q_full, (tiles - 1) & 1, &no_abort, tmo, nullptr, 0);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      constexpr uint32_t idesc_s = make_idesc(kBlockM, kBlockN, 1, false);
      constexpr uint32_t idesc_o = make_idesc(kBlockM, D, 1, true);
      uint32_t kv_iter = 0, s_iter = 0, p_iter = 0;
      int tiles = 0;
      bool ok = true;
      for (int round = 0; ok; ++round) {
        const int u = unit_for_round(round, p.num_units);
        if (u < 0) break;
        int bh, qb;
        unit_coords(u, p.num_qblocks, p.causal, bh, qb);
        const int nkv = num_kv_blocks(qb, p.N, p.causal);
        if (!(ok = mbar_wait(b_q_full, tiles & 1, abort_flag, tmo, p.err, 10))) break;
        uint32_t prev_st = 0, prev_use = 0;
        for (int j = 0; j <= nkv && ok; ++j) {
          uint32_t st = 0, use = 0;
          if (j < nkv) {
            // S_j = Q K_j^T into S buffer (s_iter & 1)
            st = kv_iter % NSTAGE;
            use = kv_iter / NSTAGE;
            const uint32_t b = s_iter & 1;
            if (!(ok = mbar_wait(b_k_full0 + 8 * st, use & 1, abort_flag, tmo, p.err, 11))) break;
            if (s_iter >= 2 && !(ok = mbar_wait(b_s_free0 + 8 * b, ((s_iter >> 1) - 1) & 1, abort_flag, tmo, p.err, 12)))
              break;
            tc_fence_after();
            const uint32_t d_tmem = tmem + (b ? kTmemS1 : kTmemS0);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * L::kChunkBytes + (kk & 3) * 32;
              mma_f16_ss(d_tmem, sdesc_sw128(sQ + off, 16, 1024),
                         sdesc_sw128(sK + st * L::kTileBytes + off, 16, 1024), idesc_s, kk > 0);
            }
            mma_commit(b_s_full0 + 8 * b);
            if (j == nkv - 1) mma_commit(b_q_empty);
            ++s_iter;
            ++kv_iter;
          }
          if (j >= 1) {
            // O += P_{j-1} V_{j-1}
            if (!(ok = mbar_wait(b_p_full, p_iter & 1, abort_flag, tmo, p.err, 13))) break;
            ++p_iter;
            if (!(ok = mbar_wait(b_v_full0 + 8 * prev_st, prev_use & 1, abort_flag, tmo, p.err, 14))) break;
            if (j == 1 && tiles > 0 && !(ok = mbar_wait(b_o_free, (tiles - 1) & 1, abort_flag, tmo, p.err, 15)))
              break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kBlockN / 16; ++kk) {
              mma_f16_ts(tmem + kTmemO, tmem + kTmemP + kk * 8,
                         sdesc_sw128(sV + prev_st * L::kTileBytes + kk * 16 * 128, L::kChunkBytes, 1024), idesc_o,
                         (j > 1 || kk > 0) ? 1u : 0u);
            }
            mma_commit(b_pv_done);
            mma_commit(b_kv_empty0 + 8 * prev_st);
          }
          prev_st = st;
          prev_use = use;
        }
        ++tiles;
      }
      // Make sure every MMA issued has completed before TMEM is released.
      mma_commit(b_drain);
      volatile int no_abort = 0;
      mbar_wait(b_drain, 0, &no_abort, tmo, nullptr, 0);
    }
  } else {
    // -------------------------------------------------------------- softmax
    const int row_in_tile = threadIdx.x;  // 0..127, = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float sl2 = p.scale_log2;
    uint32_t s_iter = 0, pv_iter = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const int u = unit_for_round(round, p.num_units);
      if (u < 0) break;
      int bh, qb;
      unit_coords(u, p.num_qblocks, p.causal, bh, qb);
      const int nkv = num_kv_blocks(qb, p.N, p.causal);
      const int row = qb * kBlockM + row_in_tile;
      float m_use = -INFINITY;  // running max in log2 units (scale folded in)
      float l = 0.f;            // running normaliser against m_use
      for (int j = 0; j < nkv; ++j) {
        const uint32_t b = s_iter & 1;
        if (!(ok = warp_wait(b_s_full0 + 8 * b, (s_iter >> 1) & 1, abort_flag, tmo, p.err, 20))) break;
        tc_fence_after();
        uint32_t sraw[kBlockN];
        tmem_ld128_wait(tmem + lane_addr + (b ? kTmemS1 : kTmemS0), sraw);
        tc_fence_before();
        mbar_arrive(b_s_free0 + 8 * b);
        ++s_iter;
        float s[kBlockN];
#pragma unroll
        for (int c = 0; c < kBlockN; ++c) s[c] = __uint_as_float(sraw[c]);
        // mask: causal (key > row) on the diagonal block, keys >= N on the tail block
        const int key0 = j * kBlockN;
        if ((p.causal && j == qb) || key0 + kBlockN > p.N) {
          const int lim_causal = p.causal ? (row - key0) : (kBlockN - 1);
          const int lim_tail = p.N - 1 - key0;
          const int lim = lim_causal < lim_tail ? lim_causal : lim_tail;
#pragma unroll
          for (int c = 0; c < kBlockN; ++c)
            if (c > lim) s[c] = -INFINITY;
        }
        float mx = s[0];
#pragma unroll
        for (int c = 1; c < kBlockN; ++c) mx = fmaxf(mx, s[c]);
        const float m_blk = mx * sl2;
        float alpha = 1.f;
        bool moved = false;
        if (m_blk > m_use + kRescaleThreshold) {
          alpha = ex2_approx(m_use - m_blk);  // 0 when m_use = -inf
          m_use = m_blk;
          moved = true;
        }
        const float m_sub = (m_use == -INFINITY) ? 0.f : m_use;
        float rs = 0.f;
        uint32_t pk[kBlockN / 2];
#pragma unroll
        for (int c = 0; c < kBlockN; c += 2) {
          const float e0 = ex2_approx(fmaf(s[c], sl2, -m_sub));
          const float e1 = ex2_approx(fmaf(s[c + 1], sl2, -m_sub));
          rs += e0 + e1;
          pk[c / 2] = pack_bf16x2(e0, e1);
        }
        l = l * alpha + rs;
        if (j >= 1) {
          // P and O are still in use by the previous P V product.
          if (!(ok = warp_wait(b_pv_done, pv_iter & 1, abort_flag, tmo, p.err, 21))) break;
          ++pv_iter;
          tc_fence_after();
          if (__any_sync(0xffffffffu, moved)) {
            // O row *= alpha (alpha = 1 for rows whose max did not move)
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t o[32];
              tmem_ld32_wait(tmem + lane_addr + kTmemO + c0, o);
#pragma unroll
              for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
              tmem_st32(tmem + lane_addr + kTmemO + c0, o);
            }
          }
        }
        tmem_st64(tmem + lane_addr + kTmemP, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(b_p_full);
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (!(ok = warp_wait(b_pv_done, pv_iter & 1, abort_flag, tmo, p.err, 22))) break;
      ++pv_iter;
      tc_fence_after();
      uint32_t oraw[D];
      if constexpr (D == 128) tmem_ld128_wait(tmem + lane_addr + kTmemO, oraw);
      else tmem_ld64_wait(tmem + lane_addr + kTmemO, oraw);
      tc_fence_before();
      mbar_arrive(b_o_free);  // the next tile's first P V may overwrite O now
      const float inv_l = 1.f / l;
      if (row < p.N) {
        uint4* dst = reinterpret_cast<uint4*>(p.o + (static_cast<size_t>(bh) * p.N + row) * D);
#pragma unroll
        for (int v = 0; v < D / 8; ++v) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = pack_bf16x2(__uint_as_float(oraw[8 * v + 2 * e]) * inv_l,
                               __uint_as_float(oraw[8 * v + 2 * e + 1]) * inv_l);
          dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        if (p.lse != nullptr) {
          // lse = ln(sum_j exp(scale * s_j)) = ln2 * (m_use + log2(l))
          p.lse[static_cast<size_t>(bh) * p.N + row] = (m_use + lg2_approx(l)) * 0.69314718055994530942f;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int NSTAGE>
constexpr size_t fwd_smem_bytes() {
  return 1024 /*alignment slack*/ + SmemLayout<D>::kTileBytes * (1 + 2 * NSTAGE) + 8 * (10 + 3 * NSTAGE) + 16;
}

}  // namespace attn
