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
// Blackwell mapping, one persistent CTA per SM.  A work unit is a pair of
// 128-row query tiles (tile 0 = rows 256p..256p+127, tile 1 = the next 128) of one
// (batch, head); both tiles stream the same K/V blocks:
//   warps 0-3   softmax of tile 0 (thread t owns row t = TMEM lane t)
//   warps 4-7   softmax of tile 1
//   warp  8     producer: TMA loads of the two Q tiles and of the K and V
//               blocks into two rings of shared-memory stages
//   warp  9     MMA warp (one elected lane issues): S_t = Q_t K_j^T, O_t += P_t V_j
//   warps 10-11 FP8 only: convert each e4m3 V block to f16 in shared memory
// The MMA warp interleaves the tiles -- P0 V_j, S0 = Q0 K_{j+1}^T, P1 V_j,
// S1 = Q1 K_{j+1}^T -- so that the softmax of one tile runs while the tensor
// core works on the other.
//
// TMEM (512 columns x 128 lanes of 32 bit):  S_0 at 0, S_1 at 128 (fp32 scores),
// O_0 at 256, O_1 at 256 + D (fp32 accumulators).  P_t (16-bit, two per column)
// overwrites the first 64 columns of S_t once the scores are in registers; the
// next S_t = Q_t K^T is issued after O_t += P_t V, and tcgen05.mma operations
// issued by one thread execute in issue order, so P_t is consumed before S_t is
// rewritten.
//
// Synchronisation (mbarriers):
//   q_full/q_empty        the two Q tiles of a unit (TMA -> MMA -> TMA)
//   k_full/k_empty[st]    K ring (TMA -> MMA; freed after the last S using it)
//   v_full/v_empty[st]    V ring (TMA -> MMA, or -> converter for FP8; BF16 frees
//                         a stage right after tile 1's P V, before the next S)
//   c_full/c_empty[b]     FP8: f16 copy of V (converter -> MMA -> converter)
//   s_full[t]   MMA -> softmax: S_t,j ready; since it is committed after
//               O_t += P_t,j-1 V_j-1, it also means O_t and P_t are free
//   pa_full[t]  softmax -> MMA: the first half of P_t,j (keys 0-63) written (and
//               O_t rescaled if needed); its half of P V may start
//   p_full[t]   softmax -> MMA: all of P_t,j written
//   pv_done[t]  MMA -> softmax: the unit's last P_t V product has completed
//   o_free[t]   softmax -> MMA: the epilogue has read O_t
//   ost_ready[t], ost_free[t]  (kTmaO) epilogue threads -> the warpgroup's
//               storing thread: a 64-column chunk of bf16 O_t is in the staging
//               buffer; storing thread -> epilogue threads: its TMA store has read
//               the buffer
//
// Row max: the scores come out of TMEM with tcgen05.ld.red .max (a Blackwell
// Ultra form), which returns each row's maximum with the load, so a block
// without masked keys spends no instructions on it; masked blocks (the causal
// diagonal, keys past N) take the maximum of the visible scores in registers.
//
// Epilogue: O_t / l to bf16.  kTmaO instances (non-causal BF16 launches) stage
// each 64-column chunk in shared memory (128-byte swizzle) and store it with one
// TMA tensor store per chunk (rows past N clipped by the tensor map); the others
// store each thread's row directly in 16-byte pieces.
//
// Block-scaled FP8 variant (kFp8): Q, K, V are e4m3 with one fp32 scale per
// (batch, head, 128-token block) -- the block quantisation and FP8 tensor-core
// path of the FlashAttention-3 notes in the news article, section 1.
// S = Q8 K8^T runs as tcgen05.mma kind::f8f6f4 and the true score is
// s_q * s_k[j] * S, so s_q * s_k[j] is folded into the exponent multiplier.
// P V runs as kind::f16: the e4m3 V codes are converted exactly to f16 in shared
// memory and P is rounded to f16 (an e4m3 P loses too much precision once V has
// outlier channels).  The V block scale and a 2^6 pre-scale are folded into the
// exponent offset, P' = 2^(x - m + 6 + log2(s_v[j] / max s_v)) <= 2^14, and at
// the end O = O' * max s_v / (64 l).
//
// Direct-P FP4 variant (kFp4, with kFp8's e4m3 Q K^T): P V runs on the FP4
// tensor cores (kind::mxf4: e2m1 elements, one power-of-two scale per 32 keys),
// with V supplied as MXFP4 along the keys and stored transposed ([d][N/2] bytes,
// K-major, 64-byte swizzle).  P goes from scores to 4-bit codes directly (the
// FP4 FlashAttention-4 summary's Direct-P): each 32-key block of a row takes its
// scale exponent E from its largest score, E = ceil(max t), so the code of a key
// is e2m1(2^(t - E + 2)) -- one exponential and one conversion, no pass over the
// probabilities to find their block maximum and no division by the scale.  The
// running max moves in whole powers of two, so rescales are exact and the codes
// depend on the scores alone.  P (16 columns), its scales and V's scales are
// written into dead S_t columns (0..15, 32..35, 64..67); the row sum is taken
// from the codes.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace attn {

constexpr int kBlockM = 128;      // query rows per tile (= TMEM lanes)
constexpr int kBlockN = 128;      // keys per K/V block
constexpr int kTilesPerUnit = 2;  // query tiles sharing the K/V stream
constexpr int kNumThreads = 384;  // 12 warps
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kConvertWarp0 = 10;  // warps 10-11
constexpr int kConvertThreads = 64;
constexpr uint32_t kTmemCols = 512;
// Register split (setmaxnreg): the launch gives 168 registers per thread
// (65536 / 384 rounded down to a multiple of 8); the two softmax warpgroups take
// 216 and the control warpgroup keeps 72:  2*128*216 + 128*72 = 168*384.
constexpr uint32_t kRegsLaunch = 168, kRegsSoftmax = 216, kRegsControl = 72;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsControl == kRegsLaunch * kNumThreads,
              "register split must add up to the launch allocation");
// The running max is only moved when a block raises it by more than this many
// powers of two; until then exponentials are taken against the stale max and are
// at most 2^8, which the 16-bit P and the fp32 accumulators absorb.
constexpr float kRescaleThreshold = 8.0f;
constexpr float kFp8PScaleLog2 = 6.0f;
// FP8 stores P' = 2^(x - m + kFp8PScaleLog2 + ...) in f16, with x - m at most the
// threshold: the largest P' must stay below f16's largest binade (2^15).  (A
// threshold of 12 overflowed to inf; 8, 12 and 16 ran at the same speed.)
static_assert(kRescaleThreshold + kFp8PScaleLog2 <= 15.0f, "FP8 P' would overflow f16");
// Every kPolyEvery-th pair of scores of a row would take its two exponentials
// from the FMA pipe (exp2_poly2) instead of the special-function unit; 0 = all
// on the SFU.  Measured on GB300 (doubled SFU ex2 rate), every share is slower:
// B1 H32 N16384 causal d = 128: 1659 TFLOP/s at 0, 1621 at 1/8, 1556 at 1/4, 1376
// at 1/2; d = 64 1022 -> 994 -> 944 -> 741.  The polynomial costs about ten
// FMA/ALU instructions per pair against two SFU issues, and the softmax is
// bound by its instruction chain rather than by the SFU's throughput.
#ifndef ATTN_POLY_EXP2_EVERY
#define ATTN_POLY_EXP2_EVERY 0
#endif
constexpr int kPolyEvery = ATTN_POLY_EXP2_EVERY;


// Direct-P FP4: TMEM columns (within S_t) of the P scales and the V^T scales
constexpr uint32_t kFp4SfaCol = 32, kFp4SfbCol = 64;

struct FwdParams {
  __nv_bfloat16* o;   // final output: [B*H, Nq, D] bf16
  float* lse;         // final output: [B*H, Nq] or nullptr
  float* o_part;      // partial output: [num_splits, B*H, Nq, D] fp32
  float* lse_part;    // partial output: [num_splits, B*H, Nq] fp32
  int BH;             // B*H
  int Nq, Nk;         // query rows and key rows per head
  int q_offset;       // causal positions: query i sits at q_offset + i,
  int k_offset;       //   key j at k_offset + j; j visible to i iff k_pos <= q_pos
  int num_kblocks;    // ceil(Nk / 128)
  int num_pairs;      // ceil(Nq / 256)
  int num_splits;     // key-block ranges per (bh, pair)
  int blocks_per_split;
  int num_units;      // BH * num_pairs * num_splits
  int causal;
  int o_align32;      // o is 32-byte aligned (set at launch)
  int order;          // unit order: kOrderHeads, kOrderZigzag or kOrderGroups (below)
  int group_heads;    // kOrderGroups: heads per group
  int sched_table;    // launched as a kTable instance (host bookkeeping)
  int pair_tail;      // head-major, unsplit: the last, partly filled round's units are
                      //   split in two key halves over the two CTAs of a cluster pair
  float scale_log2;   // scale * log2(e)
  const float* q_scale;  // FP8 only: [B*H, num_kblocks] block scales
  const float* k_scale;
  const float* v_scale;  // FP8; the Direct-P FP4 path keeps here the E8M0 scales of
                         //   V^T, 32-bit words of four bytes: [B*H, D, Nk/128]
  unsigned long long timeout_ns;
  int* err;           // device error word (first failure wins)
};

// A 128-row tile of D elements is stored as D*elem/128 column chunks of
// 128 rows x 128 bytes (the TMA box and the 128-byte swizzle atom width).
template <int D, int kElemBytes>
struct TileLayout {
  static constexpr uint32_t kChunkElems = 128 / kElemBytes;      // elements per 128-byte row
  static constexpr uint32_t kChunkBytes = kBlockM * 128;         // 128 rows x 128 bytes
  static constexpr uint32_t kChunks = D / kChunkElems;
  static constexpr uint32_t kTileBytes = kChunks * kChunkBytes;  // one 128 x D tile
  static constexpr uint32_t kMmaK = 32 / kElemBytes;             // K of one tcgen05.mma (32 bytes)
  static_assert(kChunks >= 1, "head dimension too small for the 128-byte swizzle");
};

// One round of a CTA's schedule, decoded (the unit table in shared memory).
struct SchedEntry {
  int u;  // unit id, or kNoMoreUnits / kSkipRound
  int bh, pair, split, kb0, n0, n1, role;
};
constexpr int kSchedEntries = 64;     // rounds a CTA of a kTable instance may take
constexpr int kSchedEntriesTma = 48;  // ... of a kTable instance with the O staging buffers

// Shared-memory plan of one instance: Q tiles, K ring, V ring and (FP8) the f16
// copy of V, the unit table, then the mbarriers.
template <int D, int NK, int NV, bool kFp8, bool kFp4 = false, bool kTmaO = false, bool kTable = false>
struct SmemPlan {
  using In = TileLayout<D, kFp8 ? 1 : 2>;   // Q, K, V as loaded
  using V16 = TileLayout<D, 2>;              // V operand of P V (bf16 or f16)
  static constexpr int kNumConv = (kFp8 && !kFp4) ? 2 : 0;
  // FP4: a V^T tile is D rows of 128 keys x 4 bits = 64 bytes
  static constexpr uint32_t kVTileBytes = kFp4 ? D * 64 : In::kTileBytes;
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + kTilesPerUnit * In::kTileBytes;
  static constexpr uint32_t kV = kK + NK * In::kTileBytes;
  static constexpr uint32_t kC = kV + NV * kVTileBytes;
  // TMA store of O (kTmaO): per tile a 128 x 64 bf16 staging chunk (128-byte
  // swizzle)
  static constexpr uint32_t kOst = kC + kNumConv * V16::kTileBytes;
  static constexpr uint32_t kOstChunkBytes = kBlockM * 128;
  // the CTA's unit table (kTable instances: all its rounds, decoded)
  static constexpr int kSchedN = kTable ? (kTmaO ? kSchedEntriesTma : kSchedEntries) : 0;
  static constexpr uint32_t kSched = kOst + (kTmaO ? kTilesPerUnit * kOstChunkBytes : 0);
  static constexpr uint32_t kBars = kSched + kSchedN * sizeof(SchedEntry);
  static constexpr int kNumBars = 21 + 2 * NK + 2 * NV + 2 * kNumConv;
  static constexpr size_t kBytes = 1024 /*alignment slack*/ + kBars + 8 * kNumBars + 16;
  static_assert(kBytes <= 232448, "shared memory plan exceeds 227 KB");
};

// Run order (FwdParams::order):
//   kOrderHeads   head-major: the units of a head are adjacent, so concurrently
//                 running units share K/V in L2; under the causal mask each head's
//                 pairs run from the heaviest (last rows) to the lightest; the
//                 key-range splits of a pair are adjacent.
//   kOrderZigzag  causal, unsplit: heavy+light pairs combined, head-major (see
//                 unit_for_round).
//   kOrderGroups  causal, unsplit: the heads in groups of group_heads; a group's
//                 units pair-major, heaviest first, dealt back and forth over the
//                 CTAs (close to longest-job-first balance); the groups run one
//                 after another, each starting from the other end of the grid, so
//                 that the CTAs running at a time share one or two groups' K/V in
//                 L2.  One group of all heads is plain pair-major order.
// The host picks the order and the group size by predicting each candidate's
// balance with the same functions (`unit_for_round`, `unit_info`).
constexpr int kOrderHeads = 0, kOrderZigzag = 1, kOrderGroups = 2;
constexpr long long kPairOrderMaxKvBytes = 64ll << 20;
struct UnitInfo {
  int bh, pair, split;
  int kb0;   // first K/V block of the unit's key range
  int n[2];  // K/V blocks tile 0 / tile 1 visit (n[1] >= n[0])
  int role;  // pair tail: 0 a whole unit, 1 the first key half (merges), 2 the second (sends)
};

__host__ __device__ __forceinline__ UnitInfo unit_info(int u, const FwdParams& p, int role = 0) {
  UnitInfo ui;
  const int per_head = p.num_pairs * p.num_splits;
  ui.bh = u / per_head;
  const int r = u - ui.bh * per_head;
  const int pr = r / p.num_splits;
  ui.split = r - pr * p.num_splits;
  ui.pair = p.causal ? (p.num_pairs - 1 - pr) : pr;
  ui.role = role;
  ui.kb0 = ui.split * p.blocks_per_split;
  int kb_end = ui.kb0 + p.blocks_per_split;
  if (kb_end > p.num_kblocks) kb_end = p.num_kblocks;
  if (role != 0) {  // pair tail (one split): the first or the second half of the key blocks
    const int h = (p.num_kblocks + 1) / 2;
    ui.kb0 = role == 1 ? 0 : h;
    kb_end = role == 1 ? h : p.num_kblocks;
  }
  for (int t = 0; t < kTilesPerUnit; ++t) {
    int hi = kb_end;
    if (p.causal) {
      // the last key visible to the tile's last existing row
      int last_row = (2 * ui.pair + t) * kBlockM + kBlockM - 1;
      if (last_row > p.Nq - 1) last_row = p.Nq - 1;
      const int kmax = p.q_offset + last_row - p.k_offset;
      const int lim = kmax < 0 ? 0 : kmax / kBlockN + 1;
      if (hi > lim) hi = lim;
    }
    ui.n[t] = hi > ui.kb0 ? hi - ui.kb0 : 0;
  }
  return ui;
}

constexpr int kNoMoreUnits = -1;
constexpr int kSkipRound = -2;

// Rounds that grid position cc (of G) takes when U units are dealt back and
// forth: round r holds unit r G + cc on even rounds and r G + G - 1 - cc on odd.
__host__ __device__ __forceinline__ int dealt_rounds(int U, int cc, int G) {
  const int full = U / G;
  const int off = (full & 1) ? (G - 1 - cc) : cc;
  return full + (off < U - full * G ? 1 : 0);
}

// The unit CTA c of a grid of G processes in its `round`-th iteration,
// kNoMoreUnits when it is done, or kSkipRound for an iteration without a unit
// (every role skips it).
//
// kOrderZigzag: pair p of a head costs about 4p+3 K/V blocks, so the heavy pair
// P-1-k and the light pair k together cost the same for every k.  Combined unit
// j = (head, k) goes to CTA j mod G; the CTA runs its heavy pair in the even
// iteration and its light pair in the odd one (an odd pair count leaves the
// middle pair alone).  Combined units of one head are adjacent, so the CTAs
// running at a time share a few heads' K/V in L2.
// kOrderGroups: group g (heads g Hg ..) holds Hg P units, position q = pr Hg + h
// for the pr-th heaviest pair of its h-th head; the group is dealt back and forth
// from grid position c (even groups) or G - 1 - c (odd groups), so CTA c takes
// dealt_rounds(.., c) + dealt_rounds(.., G - 1 - c) rounds per two full groups.
// kOrderHeads: position c of each round on even rounds and the mirror position
// on odd rounds (the units of a head are adjacent).
// kGroups = false leaves kOrderGroups out (instances that never run it).
template <bool kGroups = true>
__host__ __device__ __forceinline__ int unit_for_round(int round, const FwdParams& p, int G, int c) {
  if (p.order == kOrderZigzag) {
    const int half = (p.num_pairs + 1) >> 1;
    const int k = (round >> 1) * G + c;
    if (k >= p.BH * half) return kNoMoreUnits;
    const int bh = k / half;
    const int cc = k - bh * half;
    const int heavy = p.num_pairs - 1 - cc;
    if ((round & 1) && heavy == cc) return kSkipRound;
    const int pair = (round & 1) ? cc : heavy;
    return bh * p.num_pairs + (p.num_pairs - 1 - pair);  // unit id as unit_info decodes it
  }
  if (kGroups && p.order == kOrderGroups) {
    const int hg = p.group_heads;
    const int num_groups = (p.BH + hg - 1) / hg;
    const int full_units = hg * p.num_pairs;
    const int n0 = dealt_rounds(full_units, c, G), n1 = dealt_rounds(full_units, G - 1 - c, G);
    if (n0 + n1 == 0) return kNoMoreUnits;
    int g = 2 * (round / (n0 + n1));
    int r = round - (g >> 1) * (n0 + n1);
    if (r >= n0) {
      r -= n0;
      ++g;
    }
    if (g >= num_groups) return kNoMoreUnits;
    const int heads = (p.BH - g * hg) < hg ? (p.BH - g * hg) : hg;  // the last group may be smaller
    const int cc = (g & 1) ? (G - 1 - c) : c;
    if (heads < hg && r >= dealt_rounds(heads * p.num_pairs, cc, G)) return kNoMoreUnits;
    const int q = r * G + ((r & 1) ? (G - 1 - cc) : cc);
    const int pr = q / heads;  // 0: the heaviest pair
    const int bh = g * hg + (q - pr * heads);
    return bh * p.num_pairs + pr;
  }
  if (p.pair_tail) {
    // full rounds as below; then unit full G + k for the CTA pair (2k, 2k+1)
    const int full = p.num_units / G;
    if (round > full) return kNoMoreUnits;
    if (round == full) {
      const int pos = full * G + (c >> 1);
      return pos < p.num_units ? pos : kNoMoreUnits;
    }
  }
  const int pos = round * G + ((round & 1) ? (G - 1 - c) : c);
  return pos < p.num_units ? pos : kNoMoreUnits;
}

// The pair-tail role of CTA c in `round` (UnitInfo::role): 1 or 2 in the last
// round of a pair-tail launch (the even CTA of the pair takes the first key half
// and merges, the odd one the second half and sends), else 0.
__host__ __device__ __forceinline__ int tail_role(int round, const FwdParams& p, int G, int c) {
  if (!p.pair_tail || p.order != kOrderHeads || round != p.num_units / G) return 0;
  return (p.num_units / G) * G + (c >> 1) < p.num_units ? 1 + (c & 1) : 0;
}

// The unit of the CTA's `round`-th iteration and its decoded info.  kTable
// instances (kN > 0) read it from the table the CTA fills in its prologue (all
// threads, one round each), so that no role spends the schedule's integer
// divisions on its path from one unit to the next; the host launches them only
// when every CTA's rounds fit in the table.  The others compute it here, and
// the host gives them only the head-major and zigzag orders, whose arithmetic
// is short.
template <int kN, bool kTail = false>
__device__ __forceinline__ int next_unit(int round, const SchedEntry* tab, const FwdParams& p, UnitInfo& ui) {
  if constexpr (kN > 0) {
    if (round >= kN) return kNoMoreUnits;
    const SchedEntry e = tab[round];
    ui.bh = e.bh;
    ui.pair = e.pair;
    ui.split = e.split;
    ui.kb0 = e.kb0;
    ui.n[0] = e.n0;
    ui.n[1] = e.n1;
    ui.role = e.role;
    return e.u;
  } else {
    const int u = unit_for_round<false>(round, p, gridDim.x, blockIdx.x);
    if (u >= 0) ui = unit_info(u, p, kTail ? tail_role(round, p, gridDim.x, blockIdx.x) : 0);
    return u;
  }
}

// Largest of 128 scores: four independent chains of three-input max.
__device__ __forceinline__ float row_max128(const float (&s)[kBlockN]) {
  float a0 = fmaxf(s[0], s[1]), a1 = fmaxf(s[2], s[3]), a2 = fmaxf(s[4], s[5]), a3 = fmaxf(s[6], s[7]);
#pragma unroll
  for (int c = 8; c < kBlockN; c += 8) {
    a0 = fmax3(a0, s[c], s[c + 1]);
    a1 = fmax3(a1, s[c + 2], s[c + 3]);
    a2 = fmax3(a2, s[c + 4], s[c + 5]);
    a3 = fmax3(a3, s[c + 6], s[c + 7]);
  }
  return fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
}

// A wait taken by all 32 lanes of a warp that returns the same answer on every
// lane, so that the warp stays converged for the .sync.aligned tcgen05 ops.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t timeout_ns, int* err_word, int where) {
  const bool ok = mbar_wait(bar, parity, abort_flag, timeout_ns, err_word, where);
  return __all_sync(0xffffffffu, ok);
}
// The same for a barrier the partner CTA of a cluster pair arrives on.
__device__ __forceinline__ bool warp_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                  uint64_t timeout_ns, int* err_word, int where) {
  const bool ok = mbar_wait_cluster(bar, parity, abort_flag, timeout_ns, err_word, where);
  return __all_sync(0xffffffffu, ok);
}

template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// kPartial selects the output: false = normalised bf16 O and lse (every query
// row sees key 0: no position offsets, no splits); true = per-split fp32 O and
// lse, where a tile or row may see no key at all.  kTmaO (final bf16 output
// only): O leaves through shared-memory staging and TMA stores instead of
// row-per-thread global stores.
template <int D, int NK, int NV, bool kFp8, bool kPartial, bool kFp4 = false, bool kTmaO = false,
          bool kTable = false, bool kPairTail = false>
__global__ void __launch_bounds__(kNumThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_o,
                const FwdParams p) {
  static_assert(!kFp4 || (kFp8 && D == 128 && !kPartial), "Direct-P FP4: e4m3 Q K^T, d = 128, final output");
  static_assert(!kTmaO || !kPartial, "the TMA store serves the final bf16 output");
  using Plan = SmemPlan<D, NK, NV, kFp8, kFp4, kTmaO, kTable>;
  static_assert(!kPairTail || (!kPartial && !kFp4 && (kTable || kFp8)),
                "the pair tail serves BF16 table launches and FP8 launches");
  using L = typename Plan::In;
  using LV = typename Plan::V16;
  constexpr uint32_t kTmemS[2] = {0, 128};
  constexpr uint32_t kTmemO[2] = {256, 256 + D};

  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle atoms.
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);

  const uint32_t sQ = base + Plan::kQ;  // tile t at sQ + t * kTileBytes
  const uint32_t sK = base + Plan::kK;
  const uint32_t sV = base + Plan::kV;
  const uint32_t sC = base + Plan::kC;  // FP8: f16 V buffers
  const uint32_t sOst = base + Plan::kOst;  // + t * kOstChunkBytes: O staging of tile t
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Plan::kBars);
  const uint32_t b_q_full = smem_u32(&bars[0]);
  const uint32_t b_q_empty = smem_u32(&bars[1]);
  const uint32_t b_drain = smem_u32(&bars[2]);
  const uint32_t b_s_full = smem_u32(&bars[4]);    // + 8 t
  const uint32_t b_p_full = smem_u32(&bars[6]);    // + 8 t
  const uint32_t b_pv_done = smem_u32(&bars[8]);   // + 8 t
  const uint32_t b_o_free = smem_u32(&bars[10]);   // + 8 t
  const uint32_t b_k_full = smem_u32(&bars[12]);   // + 8 stage
  const uint32_t b_k_empty = smem_u32(&bars[12 + NK]);
  const uint32_t b_v_full = smem_u32(&bars[12 + 2 * NK]);
  const uint32_t b_v_empty = smem_u32(&bars[12 + 2 * NK + NV]);
  const uint32_t b_c_full = smem_u32(&bars[12 + 2 * NK + 2 * NV]);  // + 8 b (FP8)
  const uint32_t b_c_empty = b_c_full + 8 * Plan::kNumConv;
  const uint32_t b_pa_full = b_c_empty + 8 * Plan::kNumConv;  // + 8 t: first half of P_t written
  const uint32_t b_ost_ready = b_pa_full + 8 * kTilesPerUnit;   // + 8 t: staging chunk of tile t written
  const uint32_t b_ost_free = b_ost_ready + 8 * kTilesPerUnit;  // + 8 t: ... read by its TMA store
  // pair tail: (+ 8 t) the partner's rows of tile t are in this CTA's shared memory;
  // the partner's shared memory is free for this CTA's rows
  const uint32_t b_data_ready = b_ost_free + 8 * kTilesPerUnit;
  const uint32_t b_recv_ready = b_data_ready + 8 * kTilesPerUnit;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bars[Plan::kNumBars]);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t tmo = p.timeout_ns;

  if (threadIdx.x == 0) {
    mbar_init(b_q_full, 1);
    mbar_init(b_q_empty, 1);
    mbar_init(b_drain, 1);
    for (int t = 0; t < kTilesPerUnit; ++t) {
      mbar_init(b_s_full + 8 * t, 1);
      mbar_init(b_p_full + 8 * t, 128);
      mbar_init(b_pv_done + 8 * t, 1);
      mbar_init(b_o_free + 8 * t, 128);
      mbar_init(b_pa_full + 8 * t, 128);
      mbar_init(b_ost_ready + 8 * t, 128);
      mbar_init(b_ost_free + 8 * t, 1);
      mbar_init(b_data_ready + 8 * t, 128);
    }
    for (int s = 0; s < NK; ++s) {
      mbar_init(b_k_full + 8 * s, 1);
      mbar_init(b_k_empty + 8 * s, 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(b_v_full + 8 * s, 1);
      mbar_init(b_v_empty + 8 * s, Plan::kNumConv > 0 ? kConvertThreads : 1);
    }
    for (int b = 0; b < Plan::kNumConv; ++b) {
      mbar_init(b_c_full + 8 * b, kConvertThreads);
      mbar_init(b_c_empty + 8 * b, 1);
    }
    mbar_init(b_recv_ready, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
    if constexpr (kTmaO) prefetch_tmap(&tmap_o);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  SchedEntry* sched = reinterpret_cast<SchedEntry*>(smem + Plan::kSched);
  for (int i = threadIdx.x; i < Plan::kSchedN; i += kNumThreads) {
    SchedEntry e{};
    e.u = unit_for_round(i, p, gridDim.x, blockIdx.x);
    e.role = tail_role(i, p, gridDim.x, blockIdx.x);
    if (e.u >= 0) {
      const UnitInfo ui = unit_info(e.u, p, e.role);
      e.bh = ui.bh;
      e.pair = ui.pair;
      e.split = ui.split;
      e.kb0 = ui.kb0;
      e.n0 = ui.n[0];
      e.n1 = ui.n[1];
    }
    sched[i] = e;
  }
  tc_fence_before();
  __syncthreads();
  // pair tail: the partner's barriers are initialised before anyone arrives on them
  if constexpr (kPairTail) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8) {
    setmaxnreg_dec<kRegsControl>();
    if (warp == kProducerWarp && lane == 0) {
      // ---------------------------------------------------------------- TMA
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      uint32_t gk = 0, gv = 0;  // K and V blocks issued so far
      int units = 0, q_issued = 0;  // units with work, Q loads issued
      bool ok = true;
      for (int round = 0; ok; ++round) {
        UnitInfo ui;
        const int u = next_unit<Plan::kSchedN, kPairTail>(round, sched, p, ui);
        if (u == kNoMoreUnits) break;
        if (u == kSkipRound) continue;
        const int nkv = ui.n[1];
        if (nkv == 0) continue;  // no visible keys: the softmax warps write the empty result
        if (units > 0 && !(ok = mbar_wait(b_q_empty, (units - 1) & 1, abort_flag, tmo, p.err, 1))) break;
        mbar_arrive_expect_tx(b_q_full, kTilesPerUnit * L::kTileBytes);
        for (int t = 0; t < kTilesPerUnit; ++t)
          for (int c = 0; c < (int)L::kChunks; ++c)
            tma_load_3d(sQ + t * L::kTileBytes + c * L::kChunkBytes, &tmap_q, b_q_full, c * L::kChunkElems,
                        (2 * ui.pair + t) * kBlockM, ui.bh, pol_q);
        ++q_issued;
        for (int j = 0; j < nkv; ++j) {
          const int key0 = (ui.kb0 + j) * kBlockN;
          const uint32_t sk = gk % NK, uk = gk / NK;
          if (uk > 0 && !(ok = mbar_wait(b_k_empty + 8 * sk, (uk - 1) & 1, abort_flag, tmo, p.err, 2))) break;
          mbar_arrive_expect_tx(b_k_full + 8 * sk, L::kTileBytes);
          for (int c = 0; c < (int)L::kChunks; ++c)
            tma_load_3d(sK + sk * L::kTileBytes + c * L::kChunkBytes, &tmap_k, b_k_full + 8 * sk,
                        c * L::kChunkElems, key0, ui.bh, pol_kv);
          ++gk;
          const uint32_t sv = gv % NV, uv = gv / NV;
          if (uv > 0 && !(ok = mbar_wait(b_v_empty + 8 * sv, (uv - 1) & 1, abort_flag, tmo, p.err, 3))) break;
          mbar_arrive_expect_tx(b_v_full + 8 * sv, Plan::kVTileBytes);
          if constexpr (kFp4) {
            // V^T: the block's 64 bytes of keys in every one of the D rows
            tma_load_3d(sV + sv * Plan::kVTileBytes, &tmap_v, b_v_full + 8 * sv, key0 / 2, 0, ui.bh, pol_kv);
          } else {
            for (int c = 0; c < (int)L::kChunks; ++c)
              tma_load_3d(sV + sv * L::kTileBytes + c * L::kChunkBytes, &tmap_v, b_v_full + 8 * sv,
                          c * L::kChunkElems, key0, ui.bh, pol_kv);
          }
          ++gv;
        }
        ++units;
      }
      // Tail: every copy issued has landed and every consumer that frees a stage
      // has arrived before the CTA may exit.  Waits are bounded.
      if (ok) {
        for (uint32_t i = (gk > NK ? gk - NK : 0); i < gk; ++i)
          mbar_wait(b_k_empty + 8 * (i % NK), (i / NK) & 1, abort_flag, tmo, p.err, 4);
        for (uint32_t i = (gv > NV ? gv - NV : 0); i < gv; ++i)
          mbar_wait(b_v_empty + 8 * (i % NV), (i / NV) & 1, abort_flag, tmo, p.err, 5);
        if (units > 0) mbar_wait(b_q_empty, (units - 1) & 1, abort_flag, tmo, p.err, 6);
      } else {
        // Error path: wait (bounded, ignoring the abort flag) for our own copies.
        volatile int no_abort = 0;
        for (uint32_t i = (gk > NK ? gk - NK : 0); i < gk; ++i)
          mbar_wait(b_k_full + 8 * (i % NK), (i / NK) & 1, &no_abort, tmo, nullptr, 0);
        for (uint32_t i = (gv > NV ? gv - NV : 0); i < gv; ++i)
          mbar_wait(b_v_full + 8 * (i % NV), (i / NV) & 1, &no_abort, tmo, nullptr, 0);
        if (q_issued > 0) mbar_wait(b_q_full, (q_issued - 1) & 1, &no_abort, tmo, nullptr, 0);
      }
    } else if (warp == kMmaWarp) {
      // ---------------------------------------------------------------- MMA
      // The whole warp runs this role in warp-uniform control flow; one elected
      // lane issues each MMA and commit.
      // S: bf16 (kind::f16, format 1) or e4m3 (kind::f8f6f4, format 0).
      // P V: kind::f16 with bf16 (BF16 path) or f16 (FP8 path: format 0) operands.
      constexpr uint32_t idesc_s = make_idesc(kBlockM, kBlockN, kFp8 ? 0u : 1u, false);
      constexpr uint32_t idesc_o = make_idesc(kBlockM, D, kFp8 ? 0u : 1u, true);
      uint32_t g = 0;
      uint32_t p_iter[2] = {0, 0};
      int units = 0;
      bool ok = true;
      // S_t = Q_t K^T for the K block in stage sk: K steps of 32 bytes, four per
      // 128-byte swizzled row, then on to the next column chunk.
      auto issue_s = [&](int t, uint32_t sk) {
        const uint32_t d_tmem = tmem + kTmemS[t];
        // descriptor low words of step 0; step kk adds its byte offset >> 4 (the
        // address field is 14 bits of address >> 4 and shared memory stays below
        // 2^18 bytes, so the sum never carries into the LBO field)
        const uint32_t qa0 = sdesc_lo(sQ + t * L::kTileBytes, 16);
        const uint32_t kb0 = sdesc_lo(sK + sk * L::kTileBytes, 16);
        constexpr uint32_t hi = sdesc_hi_sw128(1024);
#pragma unroll
        for (int kk = 0; kk < D / (int)L::kMmaK; ++kk) {
          const uint32_t off = ((kk >> 2) * L::kChunkBytes + (kk & 3) * 32) >> 4;
          if constexpr (kFp8) mma_f8_ss_w(d_tmem, qa0 + off, kb0 + off, hi, idesc_s, kk > 0 ? 1u : 0u);
          else mma_f16_ss_w(d_tmem, qa0 + off, kb0 + off, hi, idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(b_s_full + 8 * t);
      };
      // O_t (+)= P_t V with the 16-bit V tile at v_base: P_t from TMEM (two keys
      // per column), V MN-major, 16 key rows of 128 bytes per step, column chunks
      // kChunkBytes apart.
      // (16-bit P) `half` selects the keys: 0 = 0..63, 1 = 64..127, -1 = all.
      auto issue_pv = [&](int t, uint32_t v_base, bool accumulate, int half) {
        if constexpr (kFp4) {
          // P_t (e2m1, S_t columns 0..15) x V^T (K-major, 64-byte swizzle): two
          // K = 64 steps of 32 bytes; scale words of P and V in S_t's columns too
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            mma_mxf4_ts(tmem + kTmemO[t], tmem + kTmemS[t] + 8 * kk, sdesc_sw64(v_base + 32 * kk, 512),
                        make_idesc_mxf4(kBlockM, D, 2 * kk), tmem + kTmemS[t] + kFp4SfaCol,
                        tmem + kTmemS[t] + kFp4SfbCol, (accumulate || kk > 0) ? 1u : 0u);
        } else {
          const uint32_t vb0 = sdesc_lo(v_base, LV::kChunkBytes);
          constexpr uint32_t hi = sdesc_hi_sw128(1024);
          const int kk0 = half == 1 ? kBlockN / 32 : 0;
          const int kk1 = half == 0 ? kBlockN / 32 : kBlockN / 16;
#pragma unroll
          for (int kk = 0; kk < kBlockN / 16; ++kk)
            if (kk >= kk0 && kk < kk1)
              mma_f16_ts_w(tmem + kTmemO[t], tmem + kTmemS[t] + kk * 8, vb0 + ((kk * 16 * 128) >> 4), hi, idesc_o,
                           (accumulate || kk > 0) ? 1u : 0u);
        }
      };
      int o_uses[2] = {0, 0};  // units in which tile t has written O_t
      bool merges = false;     // pair tail: this CTA receives its partner's half
      for (int round = 0; ok; ++round) {
        UnitInfo ui;
        const int u = next_unit<Plan::kSchedN, kPairTail>(round, sched, p, ui);
        if (u == kNoMoreUnits) break;
        if (u == kSkipRound) continue;
        merges = merges || ui.role == 1;
        const int n0 = ui.n[0], n1 = ui.n[1];
        if (n1 == 0) continue;
        if (!(ok = warp_wait(b_q_full, units & 1, abort_flag, tmo, p.err, 10))) break;
        {
          const uint32_t sk = g % NK;
          if (!(ok = warp_wait(b_k_full + 8 * sk, (g / NK) & 1, abort_flag, tmo, p.err, 11))) break;
          tc_fence_after();
          if (n0 > 0) issue_s(0, sk);
          issue_s(1, sk);
          mma_commit(b_k_empty + 8 * sk);
          if (n1 == 1) mma_commit(b_q_empty);
        }
        for (int j = 0; j < n1 && ok; ++j) {
          const uint32_t gj = g + j;
          const uint32_t skn = (gj + 1) % NK, phkn = ((gj + 1) / NK) & 1;
          // the 16-bit V operand of block j
          uint32_t v_base, v_bar, v_par;
          if constexpr (kFp4) {
            v_base = sV + (gj % NV) * Plan::kVTileBytes;
            v_bar = b_v_full + 8 * (gj % NV);
            v_par = (gj / NV) & 1;
          } else if constexpr (kFp8) {
            v_base = sC + (gj & 1) * LV::kTileBytes;
            v_bar = b_c_full + 8 * (gj & 1);
            v_par = (gj >> 1) & 1;
          } else {
            v_base = sV + (gj % NV) * L::kTileBytes;
            v_bar = b_v_full + 8 * (gj % NV);
            v_par = (gj / NV) & 1;
          }
          // Operands that arrived long ago are checked first, off the path from a
          // ready P to its P V product: V_j (both tiles) and K_{j+1} (next Q K^T).
          if (!(ok = warp_wait(v_bar, v_par, abort_flag, tmo, p.err, 14))) break;
          if (j + 1 < n1 && !(ok = warp_wait(b_k_full + 8 * skn, phkn, abort_flag, tmo, p.err, 17))) break;
          for (int t = 0; t < kTilesPerUnit; ++t) {
            const int nt = t == 0 ? n0 : n1;
            if (j >= nt || !ok) continue;
            if (j == 0) {
              // O_t is overwritten: the epilogue of its previous unit must have read it
              if (o_uses[t] > 0 &&
                  !(ok = warp_wait(b_o_free + 8 * t, (o_uses[t] - 1) & 1, abort_flag, tmo, p.err, 15 + t)))
                break;
              ++o_uses[t];
            }
            if constexpr (!kFp4) {
              // the first half of P_t is written before the second is computed, so
              // its half of P V runs while the softmax works on the rest
              if (!(ok = warp_wait(b_pa_full + 8 * t, p_iter[t] & 1, abort_flag, tmo, p.err, 18 + t))) break;
              tc_fence_after();
              issue_pv(t, v_base, j > 0, 0);
            }
            if (!(ok = warp_wait(b_p_full + 8 * t, p_iter[t] & 1, abort_flag, tmo, p.err, 12 + t))) break;
            ++p_iter[t];
            tc_fence_after();
            if constexpr (kFp4) issue_pv(t, v_base, j > 0, -1);
            else issue_pv(t, v_base, true, 1);
            // tile 1 is the last user of V_j and K_{j+1}.  BF16: V_j's stage is
            // released as soon as P_1 V_j completes, ahead of the next Q K^T, so
            // that V_{j+2} starts loading earlier (d = 128 +1.8%); FP8 releases
            // its f16 copy after the Q K^T (earlier was 2% slower).
            constexpr bool kEarlyV = !kFp8;
            if (kEarlyV && t == 1) mma_commit(b_v_empty + 8 * (gj % NV));
            if (j + 1 < nt) issue_s(t, skn);
            if (j == nt - 1) mma_commit(b_pv_done + 8 * t);
            if (t == 1) {
              if constexpr (!kEarlyV) {
                if constexpr (Plan::kNumConv > 0) mma_commit(b_c_empty + 8 * (gj & 1));
                else mma_commit(b_v_empty + 8 * (gj % NV));
              }
              if (j + 1 < nt) {
                mma_commit(b_k_empty + 8 * skn);
                if (j + 1 == n1 - 1) mma_commit(b_q_empty);
              }
            }
          }
        }
        g += n1;
        ++units;
      }
      // Every MMA issued has completed before TMEM is released.
      mma_commit(b_drain);
      volatile int no_abort = 0;
      const bool drained = warp_wait(b_drain, 0, &no_abort, tmo, nullptr, 0);
      if constexpr (kPairTail) {
        // The CTA's last unit was its pair-tail half: no MMA reads and no TMA load
        // writes the Q, K and V regions any more, so the partner may write its rows
        // there (the softmax warps only read them after the partner's arrival).
        if (merges && drained && (threadIdx.x & 31) == 0)
          mbar_arrive_cluster(mapa_shared(b_recv_ready, cluster_ctarank() ^ 1u));
        __syncwarp();
      }
    } else if (Plan::kNumConv > 0 && warp >= kConvertWarp0) {
      // ------------------------------------------------- FP8: V e4m3 -> f16
      // Each thread converts 16 of the 1024 16-byte units of a V block (128 key
      // rows x 128 e4m3): the 16 codes of a unit become 32 bytes of f16 in the
      // MN-major, 128-byte-swizzled layout the P V MMA reads (two column chunks
      // of 64 channels).  Codes are exact in f16.
      const int ct = threadIdx.x - kConvertWarp0 * 32;  // 0..63
      uint32_t g = 0;
      bool ok = true;
      for (int round = 0; ok; ++round) {
        UnitInfo ui;
        const int u = next_unit<Plan::kSchedN, kPairTail>(round, sched, p, ui);
        if (u == kNoMoreUnits) break;
        if (u == kSkipRound) continue;
        const int nkv = ui.n[1];
        for (int j = 0; j < nkv && ok; ++j, ++g) {
          const uint32_t sv = g % NV, b = g & 1;
          if (!(ok = mbar_wait(b_v_full + 8 * sv, (g / NV) & 1, abort_flag, tmo, p.err, 30))) break;
          if (g >= 2 && !(ok = mbar_wait(b_c_empty + 8 * b, ((g >> 1) - 1) & 1, abort_flag, tmo, p.err, 31)))
            break;
          const uint8_t* src = smem + Plan::kV + sv * L::kTileBytes;
          uint8_t* dst = smem + Plan::kC + b * LV::kTileBytes;
#pragma unroll 4
          for (int it = 0; it < 16; ++it) {
            const int idx = ct + kConvertThreads * it;  // 0..1023
            const int r = idx >> 3;                     // key row
            const int lu = idx & 7;                     // logical unit: channels 16 lu .. 16 lu + 15
            const uint4 in = *reinterpret_cast<const uint4*>(src + r * 128 + ((lu ^ (r & 7)) << 4));
            const uint32_t w[4] = {in.x, in.y, in.z, in.w};
            uint32_t h[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              h[2 * e] = cvt_e4m3x2_to_f16x2(static_cast<uint16_t>(w[e] & 0xffffu));
              h[2 * e + 1] = cvt_e4m3x2_to_f16x2(static_cast<uint16_t>(w[e] >> 16));
            }
            const int chunk = lu >> 2;    // channels 0-63 / 64-127
            const int x0 = (lu & 3) * 2;  // first 16-byte f16 unit of the pair
            uint8_t* rowp = dst + chunk * LV::kChunkBytes + r * 128;
            *reinterpret_cast<uint4*>(rowp + ((x0 ^ (r & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4*>(rowp + (((x0 + 1) ^ (r & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
          }
          fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
          mbar_arrive(b_c_full + 8 * b);
          mbar_arrive(b_v_empty + 8 * sv);
        }
      }
    }
  } else {
    // -------------------------------------------------------------- softmax
    setmaxnreg_inc<kRegsSoftmax>();
    const int t = warp >> 2;                      // query tile of this warpgroup
    const int row_in_tile = threadIdx.x & 127;    // = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_addr + kTmemS[t];
    const uint32_t tO = tmem + lane_addr + kTmemO[t];
    uint32_t s_iter = 0, pv_iter = 0;
    uint32_t ost_uses = 0;  // TMA stores of O issued from this tile's staging chunk
    bool ok = true;
    for (int round = 0; ok; ++round) {
      UnitInfo ui;
      const int u = next_unit<Plan::kSchedN, kPairTail>(round, sched, p, ui);
      if (u == kNoMoreUnits) break;
      if (u == kSkipRound) continue;
      const int bh = ui.bh;
      const int qt = 2 * ui.pair + t;
      const int nkv = t == 0 ? ui.n[0] : ui.n[1];
      const int row = qt * kBlockM + row_in_tile;
      // mask limit of this row relative to a block's first key: key c of block jb is
      // visible iff c <= row_lim - jb*128 (causal) and jb*128 + c < Nk
      const int row_lim = p.causal ? (p.q_offset + row - p.k_offset) : 0x3fffffff;
      const int tile_lim = p.causal ? (p.q_offset + qt * kBlockM - p.k_offset) : 0x3fffffff;  // first row's
      // Exponent multiplier of the raw scores (log2 units); FP8 adds s_q * s_k[j].
      float c_q = p.scale_log2;
      float sv_max = 1.f;
      const float* ks_row = nullptr;
      const float* vs_row = nullptr;
      if constexpr (kFp4) {
        const size_t sb = static_cast<size_t>(bh) * p.num_kblocks;
        ks_row = p.k_scale + sb;
        c_q *= __ldg(p.q_scale + sb + (qt < p.num_kblocks ? qt : p.num_kblocks - 1));
      } else if constexpr (kFp8) {
        const size_t sb = static_cast<size_t>(bh) * p.num_kblocks;
        ks_row = p.k_scale + sb;
        vs_row = p.v_scale + sb;
        c_q *= __ldg(p.q_scale + sb + (qt < p.num_kblocks ? qt : p.num_kblocks - 1));
        sv_max = 0.f;  // largest V block scale this tile uses (scales are > 0)
        for (int jj = 0; jj < nkv; ++jj) sv_max = fmaxf(sv_max, __ldg(vs_row + ui.kb0 + jj));
      }
      // FP4: the V^T scale words this lane supplies, channel rows lane, lane + 32, ...
      // (word index into p.vt_scale; the launch checks that it fits 32 bits)
      uint32_t vts_idx = 0, vts_stride = 0;
      if constexpr (kFp4) {
        vts_stride = static_cast<uint32_t>(p.Nk / kBlockN);
        vts_idx = (static_cast<uint32_t>(bh) * D + (threadIdx.x & 31)) * vts_stride;
      }
      float m_use = -INFINITY;  // running max in log2 units (scale folded in)
      float l = 0.f;            // running normaliser against m_use
      for (int j = 0; j < nkv; ++j) {
        const int jb = ui.kb0 + j;  // K/V block index
        float cj = c_q;
        float off = 0.f;  // FP8: log2 of the pre-scale and V block-scale ratio
        if constexpr (kFp4) {
          cj *= __ldg(ks_row + jb);
        } else if constexpr (kFp8) {
          cj *= __ldg(ks_row + jb);
          off = kFp8PScaleLog2 + lg2_approx(__ldg(vs_row + jb) / sv_max);
        }
        if (!(ok = warp_wait(b_s_full + 8 * t, s_iter & 1, abort_flag, tmo, p.err, 20 + t))) break;
        ++s_iter;
        tc_fence_after();
        uint32_t sraw[kBlockN];
        // the raw scores' maxima come with the load: the row's (BF16 and FP8) or each
        // 32-key block's (Direct-P FP4)
        float s_max = -INFINITY;
        float bm[4];  // FP4: block maxima of the raw scores (cj > 0 keeps the order)
        if constexpr (kFp4) tmem_ld128_max32_wait(tS, sraw, bm);
        else tmem_ld128_max_wait(tS, sraw, s_max);
        float s[kBlockN];
#pragma unroll
        for (int c = 0; c < kBlockN; ++c) s[c] = __uint_as_float(sraw[c]);
        // mask: causal (key position > query position) and keys >= Nk
        const int key0 = jb * kBlockN;
        // the block needs a mask iff a key in it lies past the tile's first row or past Nk
        if (key0 + kBlockN - 1 > tile_lim || key0 + kBlockN > p.Nk) {
          const int lim = min(row_lim - key0, p.Nk - 1 - key0);  // keys c > lim are masked
#pragma unroll
          for (int c = 0; c < kBlockN; ++c)
            if (c > lim) s[c] = -INFINITY;
          // the maxima over the visible keys
          if constexpr (kFp4) {
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              float g4[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float* x = s + 32 * b + 8 * q;
                g4[q] = fmaxf(fmax3(x[0], x[1], x[2]), fmax3(x[3], x[4], fmax3(x[5], x[6], x[7])));
              }
              bm[b] = fmaxf(fmaxf(g4[0], g4[1]), fmaxf(g4[2], g4[3]));
            }
          } else {
            s_max = row_max128(s);
          }
        }
        if constexpr (kFp4) {
          // Direct-P.
          // E_b = ceil(max t) (base 2; -inf for a block without a visible key)
          float eb[4];
#pragma unroll
          for (int b = 0; b < 4; ++b) eb[b] = ceilf(bm[b] * cj);
          // codes e2m1(2^(t - E_b + 2)), eight per 32-bit column (key k in bits
          // 4 (k % 8)), and each block's sum of code values (exact integers, in
          // halves).  They depend on the scores alone, so they are formed before
          // the running max moves, and the scores die here.
          uint32_t w[16];
          float bsum[4];
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const float add = eb[b] > -INFINITY ? 2.f - eb[b] : 0.f;
            uint32_t sum2 = 0u;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t by[4];
#pragma unroll
              for (int e = 0; e < 8; e += 2) {
                const int c = 32 * b + 8 * q + e;
                const float2 y = ffma2(make_float2(s[c], s[c + 1]), make_float2(cj, cj), make_float2(add, add));
                by[e / 2] = cvt_e2m1x2(ex2_approx(y.x), ex2_approx(y.y));
              }
              const uint32_t word = pack_bytes4(by[0], by[1], by[2], by[3]);
              w[4 * b + q] = word;
              sum2 = e2m1x8_sum2(word, sum2);
            }
            bsum[b] = 0.5f * static_cast<float>(sum2);
          }
          const float e_max = fmaxf(fmaxf(eb[0], eb[1]), fmaxf(eb[2], eb[3]));
          float alpha = 1.f;
          bool moved = false;
          if (e_max > m_use + kRescaleThreshold) {
            alpha = exp2_int(m_use - e_max);  // a whole power of two; 0 when m_use = -inf
            m_use = e_max;
            moved = true;
          }
          if (j > 0 && __any_sync(0xffffffffu, moved)) {
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t o[32];
              tmem_ld32_wait(tO + c0, o);
#pragma unroll
              for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
              tmem_st32(tO + c0, o);
            }
          }
          // block scales 2^(E_b - 2 - m) as E8M0 bytes, and the row sum
          float rowsum = 0.f;
          uint32_t sfa = 0u;
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const bool empty = !(eb[b] > -INFINITY);
            const float rel = empty ? -INFINITY : eb[b] - 2.f - m_use;
            rowsum += bsum[b] * exp2_int(rel);
            const int sbyte = empty ? 0 : max(0, min(254, static_cast<int>(rel) + 127));
            sfa |= static_cast<uint32_t>(sbyte) << (8 * b);
          }
          l = l * alpha + rowsum;
          // P at S_t columns 0..15; columns 32..35: this row's P scales (every
          // column the MMA may read for it); 64..67: the V^T scale words of
          // channels lane + 32 c
          uint32_t sa4[4], sb4[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            sa4[c] = sfa;
            sb4[c] = __ldg(reinterpret_cast<const uint32_t*>(p.v_scale) + vts_idx + 32u * c * vts_stride + jb);
          }
          tmem_st16(tS, w);
          tmem_st4(tS + kFp4SfaCol, sa4);
          tmem_st4(tS + kFp4SfbCol, sb4);
        } else {
          const float m_blk = s_max * cj;
          float alpha = 1.f;
          bool moved = false;
          if (m_blk > m_use + kRescaleThreshold) {
            alpha = ex2_approx(m_use - m_blk);  // 0 when m_use = -inf
            m_use = m_blk;
            moved = true;
          }
          if (j > 0 && __any_sync(0xffffffffu, moved)) {
            // O_t row *= alpha (alpha = 1 for rows whose max did not move).  The
            // previous P_t V product has completed: s_full was committed after it.
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t o[32];
              tmem_ld32_wait(tO + c0, o);
#pragma unroll
              for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
              tmem_st32(tO + c0, o);
            }
          }
          // P = 2^(s * cj - m [+ off]), summed in four independent pairs of lanes
          const float m_sub = ((m_use == -INFINITY) ? 0.f : m_use) - off;
          float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                           make_float2(0.f, 0.f)};
          // In two halves of 64 keys: the first half of P is stored and announced
          // (pa_full) before the second is computed, so that its half of P V runs
          // meanwhile.
          uint32_t pk[kBlockN / 2];
#pragma unroll
          for (int c = 0; c < kBlockN; c += 2) {
            const float2 x = ffma2(make_float2(s[c], s[c + 1]), make_float2(cj, cj), make_float2(-m_sub, -m_sub));
            const float2 e = (kPolyEvery > 0 && (c >> 1) % (kPolyEvery > 0 ? kPolyEvery : 1) == kPolyEvery - 1)
                                 ? exp2_poly2(x)
                                 : make_float2(ex2_approx(x.x), ex2_approx(x.y));
            acc[(c >> 1) & 3] = fadd2(acc[(c >> 1) & 3], e);
            if constexpr (kFp8) pk[c / 2] = pack_f16x2(e.x, e.y);
            else pk[c / 2] = pack_bf16x2(e.x, e.y);
            if (c == kBlockN / 2 - 2) {
              tmem_st32(tS, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
              tmem_st_wait();
              tc_fence_before();
              mbar_arrive(b_pa_full + 8 * t);
            }
          }
          const float2 acc01 = fadd2(acc[0], acc[1]);
          const float2 acc23 = fadd2(acc[2], acc[3]);
          const float2 accs = fadd2(acc01, acc23);
          float rowsum = accs.x + accs.y;
          if constexpr (kFp8) rowsum *= ex2_approx(-off);  // back to the unscaled P
          l = l * alpha + rowsum;
          tmem_st32(tS + 32, *reinterpret_cast<const uint32_t(*)[32]>(&pk[32]));
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(b_p_full + 8 * t);
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if constexpr (!kPartial) {
        if (!(ok = warp_wait(b_pv_done + 8 * t, pv_iter & 1, abort_flag, tmo, p.err, 22 + t))) break;
        ++pv_iter;
        tc_fence_after();
        if constexpr (kPairTail) {
          // The role is read again here (from the table, a volatile load, or
          // computed), so that no register carries it through the block loop, and
          // the exchange runs right here, so that nothing is carried out of the loop
          // either (either spilled the 216-register softmax warps).
          int role;
          if constexpr (kTable) role = reinterpret_cast<volatile const SchedEntry*>(sched)[round].role;
          else role = tail_role(round, p, gridDim.x, blockIdx.x);
          if (role != 0) {
            const float osc = kFp8 ? sv_max * (1.f / 64.f) : 1.f;  // O' -> unnormalised O (FP8: pre-scale, V scales)
            // Pair tail: the odd CTA sends its half (O_t unnormalised, m, l per
            // row) into the even CTA's Q/K/V regions (FP8: and its f16 copies of
            // V); the even CTA merges the two halves the way split-K/V partials
            // merge, normalises and stores.  Row layout: [m, l, pad, pad, O_0 ..
            // O_{D-1}] in fp32, a 16-byte-aligned pitch whose 16-byte units fall in
            // different bank groups for 8 consecutive rows.  O_t moves 32 columns
            // at a time (few live registers).
            constexpr uint32_t kRowBytes = (D + 4) * 4;
            static_assert(2 * kBlockM * kRowBytes <= Plan::kOst,
                          "pair-tail rows exceed the Q, K, V (and f16 V) regions");
            const uint32_t my_row = base + Plan::kQ + (t * kBlockM + row_in_tile) * kRowBytes;
            const uint32_t peer = cluster_ctarank() ^ 1u;
            if (role == 2) {
              if (warp_wait_cluster(b_recv_ready, 0, abort_flag, tmo, p.err, 32)) {
                const uint32_t dst = mapa_shared(my_row, peer);
                st_cluster_v2(dst, m_use, l);  // (a four-wide store with two zero words spilled registers)
                for (int h = 0; h < D / 32; ++h) {
                  uint32_t oraw[32];
                  tmem_ld32_wait(tO + 32 * h, oraw);
#pragma unroll
                  for (int v = 0; v < 8; ++v)
                    st_cluster_v4(dst + 16 + (32 * h + 4 * v) * 4, __uint_as_float(oraw[4 * v]) * osc,
                                  __uint_as_float(oraw[4 * v + 1]) * osc, __uint_as_float(oraw[4 * v + 2]) * osc,
                                  __uint_as_float(oraw[4 * v + 3]) * osc);
                }
                mbar_arrive_cluster(mapa_shared(b_data_ready + 8 * t, peer));
              }
            } else if (warp_wait_cluster(b_data_ready + 8 * t, 0, abort_flag, tmo, p.err, 33 + t)) {
              const float4 ml = ld_shared_v4f(my_row);
              const float m = fmaxf(m_use, ml.x);
              const float a0 = m_use == -INFINITY ? 0.f : ex2_approx(m_use - m);
              const float a1 = ml.x == -INFINITY ? 0.f : ex2_approx(ml.x - m);
              const float lt = l * a0 + ml.y * a1;
              const float w0 = a0 * osc / lt, w1 = a1 / lt;
              uint4* dst = reinterpret_cast<uint4*>(p.o + (static_cast<size_t>(bh) * p.Nq + row) * D);
              for (int h = 0; h < D / 32; ++h) {
                uint32_t oraw[32];
                tmem_ld32_wait(tO + 32 * h, oraw);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                  const float4 x0 = ld_shared_v4f(my_row + 16 + (32 * h + 8 * v) * 4);
                  const float4 x1 = ld_shared_v4f(my_row + 16 + (32 * h + 8 * v + 4) * 4);
                  const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                  uint32_t w[4];
#pragma unroll
                  for (int e = 0; e < 4; ++e)
                    w[e] = pack_bf16x2(__uint_as_float(oraw[8 * v + 2 * e]) * w0 + xs[2 * e] * w1,
                                       __uint_as_float(oraw[8 * v + 2 * e + 1]) * w0 + xs[2 * e + 1] * w1);
                  if (row < p.Nq) dst[4 * h + v] = make_uint4(w[0], w[1], w[2], w[3]);
                }
              }
              if (row < p.Nq && p.lse != nullptr)
                p.lse[static_cast<size_t>(bh) * p.Nq + row] = (m + lg2_approx(lt)) * 0.69314718055994530942f;
            }
            continue;
          }
        }
        const float inv_l = ((kFp8 && !kFp4) ? sv_max * (1.f / 64.f) : 1.f) / l;
        // O in 64-column chunks: each thread writes its row's 128 bytes of bf16
        // into the tile's staging chunk (the 128-byte swizzle the tensor map
        // expects, which also keeps the 16-byte stores free of bank conflicts),
        // one thread stores the chunk with TMA (rows past Nq are clipped), and
        // the next chunk waits until the store has read the buffer.  The last
        // TMEM load frees O_t.
        if constexpr (kTmaO) {
        const uint32_t stage = sOst + t * Plan::kOstChunkBytes;
        const uint32_t my_row = stage + row_in_tile * 128;
        const bool issuer = (threadIdx.x & 127) == 0;
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          uint32_t oraw[64];
          tmem_ld64_wait(tO + 64 * h, oraw);
          if (h == D / 64 - 1) {
            tc_fence_before();
            mbar_arrive(b_o_free + 8 * t);  // the next unit's first P V may overwrite O_t now
          }
          if (ost_uses > 0 &&
              !(ok = warp_wait(b_ost_free + 8 * t, (ost_uses - 1) & 1, abort_flag, tmo, p.err, 28 + t)))
            break;
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16x2(__uint_as_float(oraw[8 * v + 2 * e]) * inv_l,
                                 __uint_as_float(oraw[8 * v + 2 * e + 1]) * inv_l);
            st_shared_v4(my_row + ((v ^ (row_in_tile & 7)) << 4), w[0], w[1], w[2], w[3]);
          }
          fence_proxy_async_smem();  // generic-proxy writes -> visible to the TMA engine
          mbar_arrive(b_ost_ready + 8 * t);
          if (issuer) {
            ok = mbar_wait(b_ost_ready + 8 * t, ost_uses & 1, abort_flag, tmo, p.err, 30 + t);
            if (ok) {
              tma_store_3d(&tmap_o, stage, 64 * h, qt * kBlockM, bh);
              bulk_commit_group();
              bulk_wait_read_all();
              mbar_arrive(b_ost_free + 8 * t);
            }
          }
          ok = __all_sync(0xffffffffu, ok);
          ++ost_uses;
          if (!ok) break;
        }
        if (!ok) break;
        } else {
          const size_t r = static_cast<size_t>(bh) * p.Nq + row;
          uint4* dst = reinterpret_cast<uint4*>(p.o + r * D);
#pragma unroll
          for (int h = 0; h < D / 64; ++h) {
            uint32_t oraw[64];
            tmem_ld64_wait(tO + 64 * h, oraw);
            if (h == D / 64 - 1) {
              tc_fence_before();
              mbar_arrive(b_o_free + 8 * t);
            }
            // BF16: 32-byte stores when O allows them (a warp's store then fills
            // whole 32-byte sectors of its 32 rows: B4 H16 N2048 d128 causal +3%); FP8
            // measured no gain
            if (!kFp8 && row < p.Nq && p.o_align32) {
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint32_t w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  w[e] = pack_bf16x2(__uint_as_float(oraw[16 * v + 2 * e]) * inv_l,
                                     __uint_as_float(oraw[16 * v + 2 * e + 1]) * inv_l);
                st_global_v8(dst + 8 * h + 2 * v, w);
              }
            } else if (row < p.Nq) {
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  w[e] = pack_bf16x2(__uint_as_float(oraw[8 * v + 2 * e]) * inv_l,
                                     __uint_as_float(oraw[8 * v + 2 * e + 1]) * inv_l);
                dst[8 * h + v] = make_uint4(w[0], w[1], w[2], w[3]);
              }
            }
          }
        }
        // lse = ln(sum_j exp(scale * s_j)) = ln2 * (m_use + log2(l)); consecutive
        // threads hold consecutive rows, so a warp's stores are contiguous
        const size_t r = static_cast<size_t>(bh) * p.Nq + row;
        if (row < p.Nq && p.lse != nullptr) p.lse[r] = (m_use + lg2_approx(l)) * 0.69314718055994530942f;
      } else {
        uint32_t oraw[D];
        if (nkv > 0) {
          if (!(ok = warp_wait(b_pv_done + 8 * t, pv_iter & 1, abort_flag, tmo, p.err, 22 + t))) break;
          ++pv_iter;
          tc_fence_after();
          if constexpr (D == 128) tmem_ld128_wait(tO, oraw);
          else tmem_ld64_wait(tO, oraw);
          tc_fence_before();
          mbar_arrive(b_o_free + 8 * t);
        } else {
#pragma unroll
          for (int c = 0; c < D; ++c) oraw[c] = 0u;
        }
        // A row that saw no visible key gets O = 0 and lse = -inf.
        const bool empty = !(l > 0.f);
        const float inv_l = empty ? 0.f : 1.f / l;
        if (row < p.Nq) {
          const size_t rp = (static_cast<size_t>(ui.split) * p.BH + bh) * p.Nq + row;
          float4* dst = reinterpret_cast<float4*>(p.o_part + rp * D);
#pragma unroll
          for (int v = 0; v < D / 4; ++v)
            dst[v] = make_float4(__uint_as_float(oraw[4 * v]) * inv_l, __uint_as_float(oraw[4 * v + 1]) * inv_l,
                                 __uint_as_float(oraw[4 * v + 2]) * inv_l, __uint_as_float(oraw[4 * v + 3]) * inv_l);
          p.lse_part[rp] = empty ? -INFINITY : (m_use + lg2_approx(l)) * 0.69314718055994530942f;
        }
      }
    }
    // the TMA stores of O have completed before the CTA exits
    if constexpr (kTmaO) {
      if ((threadIdx.x & 127) == 0) bulk_wait_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  // pair tail: neither CTA of a pair leaves while the other may still reach its
  // shared memory (every wait above is bounded, so both get here)
  if constexpr (kPairTail) cluster_sync();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace attn
