// C ABI of the attention library: argument validation, TMA tensor-map encoding,
// per-device set-up and kernel launches.  See include/attn.h for the contract.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/attn.h"
#include "attn_fwd_kernel.cuh"
#include "attn_merge.cuh"
#include "attn_bwd_kernel.cuh"

namespace {

using namespace attn;

// Device error word: a kernel that gives up on a bounded wait writes
// (where << 8) | kDevErrTimeout here (first failure wins).
__device__ int g_attn_err = 0;

unsigned long long g_timeout_ns = 4000000000ull;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int kMaxDevices = 64;

struct DeviceState {
  std::once_flag once;
  int status = ATTN_ERR_CUDA;
  int num_sms = 0;
  int* err_ptr = nullptr;
};
DeviceState g_dev[kMaxDevices];

EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

EncodeTiledFn get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

template <int D, int NK, int NV, bool kFp8, bool kPartial, bool kFp4 = false, bool kTmaO = false,
          bool kTable = false, bool kPairTail = false>
cudaError_t configure_kernel() {
  return cudaFuncSetAttribute(attn_fwd_kernel<D, NK, NV, kFp8, kPartial, kFp4, kTmaO, kTable, kPairTail>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(SmemPlan<D, NK, NV, kFp8, kFp4, kTmaO, kTable>::kBytes));
}

// Ring depths (K stages, V stages) per instance; shared memory holds the two Q
// tiles, the rings and, for FP8, two f16 copies of V.
#define ATTN_BF16_D64 64, 4, 4, false     // 32 KB + 4 x 16 KB + 4 x 16 KB
#define ATTN_BF16_D128 128, 2, 2, false   // 64 KB + 2 x 32 KB + 2 x 32 KB
#define ATTN_FP8_D128 128, 3, 3, true     // 32 KB + 3 x 16 KB + 3 x 16 KB + 2 x 32 KB
#define ATTN_FP4_D128 128, 4, 4, true     // Direct-P FP4: 32 KB + 4 x 16 KB + 4 x 8 KB (V^T e2m1)

template <int D, int RA, int RB>
cudaError_t configure_bwd() {
  const int bytes = static_cast<int>(BwdSmem<D, RA, RB>::kBytes);
  cudaError_t e =
      cudaFuncSetAttribute(attn_bwd_dq_kernel<D, RA, RB>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(attn_bwd_dkdv_kernel<D, RA, RB>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}
// ring depths of the backward passes (ring A: K or Q, ring B: V or dO)
#define ATTN_BWD_D64 64, 6, 4    // 2 + 10 tiles of 16 KB
#define ATTN_BWD_D128 128, 3, 2  // 2 + 5 tiles of 32 KB

// Per-device set-up on first use: architecture check, SM count, kernel
// attributes, address of the error word.  Returns ATTN_OK or an error status.
int device_setup(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  DeviceState& st = g_dev[dev];
  std::call_once(st.once, [&st, dev] {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      st.status = ATTN_ERR_CUDA;
      return;
    }
    if (major != 10 || minor != 3) {
      st.status = ATTN_ERR_ARCH;
      return;
    }
    if (configure_kernel<ATTN_BF16_D64, false>() != cudaSuccess ||
        configure_kernel<ATTN_BF16_D128, false>() != cudaSuccess ||
        configure_kernel<ATTN_BF16_D64, false, false, true>() != cudaSuccess ||
        configure_kernel<ATTN_BF16_D128, false, false, true>() != cudaSuccess ||
        configure_kernel<ATTN_BF16_D64, false, false, true, true>() != cudaSuccess ||
        configure_kernel<ATTN_BF16_D64, false, false, true, true, true>() != cudaSuccess ||
        configure_kernel<ATTN_BF16_D128, false, false, true, true, true>() != cudaSuccess ||
        configure_kernel<ATTN_BF16_D128, false, false, true, true>() != cudaSuccess ||
        configure_kernel<ATTN_BF16_D64, false, false, false, true>() != cudaSuccess ||
        configure_kernel<ATTN_BF16_D128, false, false, false, true>() != cudaSuccess ||
        configure_kernel<ATTN_BF16_D64, true>() != cudaSuccess ||
        configure_kernel<ATTN_BF16_D128, true>() != cudaSuccess ||
        configure_kernel<ATTN_FP8_D128, false>() != cudaSuccess ||
        configure_kernel<ATTN_FP8_D128, false, false, false, false, true>() != cudaSuccess ||
        configure_kernel<ATTN_FP4_D128, false, true>() != cudaSuccess ||
        configure_bwd<ATTN_BWD_D64>() != cudaSuccess || configure_bwd<ATTN_BWD_D128>() != cudaSuccess ||
        cudaGetSymbolAddress(reinterpret_cast<void**>(&st.err_ptr), g_attn_err) != cudaSuccess) {
      st.status = ATTN_ERR_CUDA;
      return;
    }
    st.status = ATTN_OK;
  });
  *dev_out = dev;
  return st.status;
}

// 3-D tiled map over a contiguous [BH, N, d] tensor: dims (d, N, BH), box
// (box_inner elements, 128 rows, 1), 128-byte swizzle, zero fill out of bounds.
int make_map(CUtensorMap* map, const void* ptr, CUtensorMapDataType dt, uint32_t elem_bytes, int d, int N,
             int BH, uint32_t box_inner) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return ATTN_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * elem_bytes,
                           static_cast<cuuint64_t>(d) * elem_bytes * static_cast<cuuint64_t>(N)};
  cuuint32_t box[3] = {box_inner, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_OVERFLOW;
}

// V^T of the Direct-P FP4 path: packed e2m1 bytes [BH][d][N/2] viewed as 3-D
// (N/2, d, BH); box = 64 bytes (128 keys) x d rows, 64-byte swizzle.
int make_map_vt4(CUtensorMap* map, const void* ptr, int d, int N, int BH) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return ATTN_ERR_CUDA;
  const cuuint64_t row = static_cast<cuuint64_t>(N) / 2;
  cuuint64_t dims[3] = {row, static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {row, row * static_cast<cuuint64_t>(d)};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(d), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_OVERFLOW;
}

// Pipelined forward over host buffers: the heads go in chunks through two slots of
// a device workspace; copy-in, kernel and copy-out run on three streams, so the
// transfers of one chunk overlap the kernel of another.
constexpr int kHostChunks = 8;  // measured: 8 beats 3, 4, 6, 12, 16 on the large workloads
constexpr int kHostSlots = 2;

struct HostPipe {
  std::mutex mu;
  bool ready = false;
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t entry = nullptr, last = nullptr;
  cudaEvent_t in_done[kHostSlots] = {}, comp_done[kHostSlots] = {}, out_done[kHostSlots] = {};
};
HostPipe g_pipe[kMaxDevices];

int pipe_setup(HostPipe& hp) {
  if (hp.ready) return ATTN_OK;
  const unsigned kEv = cudaEventDisableTiming;
  if (cudaStreamCreateWithFlags(&hp.s_in, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&hp.s_out, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&hp.entry, kEv) != cudaSuccess ||
      cudaEventCreateWithFlags(&hp.last, kEv) != cudaSuccess)
    return ATTN_ERR_CUDA;
  for (int i = 0; i < kHostSlots; ++i)
    if (cudaEventCreateWithFlags(&hp.in_done[i], kEv) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp.comp_done[i], kEv) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp.out_done[i], kEv) != cudaSuccess)
      return ATTN_ERR_CUDA;
  hp.ready = true;
  return ATTN_OK;
}

// A tensor the pipeline moves: host buffer and bytes per head (whole heads are
// contiguous in every layout the entry points take).
struct HostTensor {
  const void* in;  // host source (inputs), or null
  void* out;       // host destination (outputs), or null
  size_t per_head;
};
constexpr int kHostMaxTensors = 12;

struct HostChunking {
  int heads;          // heads per chunk (the last chunk may hold fewer)
  int chunks;
  size_t region[kHostMaxTensors];  // bytes of each tensor's region in a slot (256-byte multiples)
  size_t slot_bytes;  // all of a chunk's tensors
};
HostChunking host_chunking(int B, int H, const HostTensor* t, int nt) {
  HostChunking hc;
  const long long BH = static_cast<long long>(B) * H;
  const long long n = BH < kHostChunks ? BH : kHostChunks;
  hc.heads = static_cast<int>((BH + n - 1) / n);
  hc.chunks = static_cast<int>((BH + hc.heads - 1) / hc.heads);
  hc.slot_bytes = 0;
  for (int i = 0; i < nt; ++i) {
    hc.region[i] = (static_cast<size_t>(hc.heads) * t[i].per_head + 255) / 256 * 256;
    hc.slot_bytes += hc.region[i];
  }
  return hc;
}
// The BF16 path's tensors: Q, K, V in; O, LSE out.
int bf16_host_tensors(HostTensor* t, const void* q, const void* k, const void* v, void* o, float* lse, int N,
                      int d) {
  const size_t hb = static_cast<size_t>(N) * d * 2;
  t[0] = {q, nullptr, hb};
  t[1] = {k, nullptr, hb};
  t[2] = {v, nullptr, hb};
  t[3] = {nullptr, o, hb};
  t[4] = {nullptr, lse, static_cast<size_t>(N) * sizeof(float)};
  return 5;
}
// The FP8 path's tensors: e4m3 Q, K, V and their block scales in; O, LSE out.
int fp8_host_tensors(HostTensor* t, const void* q8, const void* k8, const void* v8, const float* qs,
                     const float* ks, const float* vs, void* o, float* lse, int N, int d) {
  const size_t hb = static_cast<size_t>(N) * d;
  const size_t sb = static_cast<size_t>((N + kBlockN - 1) / kBlockN) * sizeof(float);
  t[0] = {q8, nullptr, hb};
  t[1] = {k8, nullptr, hb};
  t[2] = {v8, nullptr, hb};
  t[3] = {qs, nullptr, sb};
  t[4] = {ks, nullptr, sb};
  t[5] = {vs, nullptr, sb};
  t[6] = {nullptr, o, 2 * hb};
  t[7] = {nullptr, lse, static_cast<size_t>(N) * sizeof(float)};
  return 8;
}
// The backward's tensors: Q, K, V, O, dO, LSE in; dQ, dK, dV out; its scratch
// (-lse log2e and -scale D per padded row) in the slot only.
int bwd_host_tensors(HostTensor* t, const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, int N, int d) {
  const size_t hb = static_cast<size_t>(N) * d * 2;
  const size_t npad = (static_cast<size_t>(N) + kBlockM - 1) / kBlockM * kBlockM;
  t[0] = {q, nullptr, hb};
  t[1] = {k, nullptr, hb};
  t[2] = {v, nullptr, hb};
  t[3] = {o, nullptr, hb};
  t[4] = {dout, nullptr, hb};
  t[5] = {lse, nullptr, static_cast<size_t>(N) * sizeof(float)};
  t[6] = {nullptr, dq, hb};
  t[7] = {nullptr, dk, hb};
  t[8] = {nullptr, dv, hb};
  t[9] = {nullptr, nullptr, 2 * npad * sizeof(float)};
  return 10;
}
// The Direct-P FP4 path's tensors: e4m3 Q, K, e2m1 V^T, the Q and K block scales and
// the E8M0 scales of V^T in; O, LSE out.
int fp4p_host_tensors(HostTensor* t, const void* q8, const void* k8, const void* vt4, const float* qs,
                      const float* ks, const uint8_t* vts, void* o, float* lse, int N, int d) {
  const size_t hb = static_cast<size_t>(N) * d;
  t[0] = {q8, nullptr, hb};
  t[1] = {k8, nullptr, hb};
  t[2] = {vt4, nullptr, hb / 2};
  t[3] = {qs, nullptr, static_cast<size_t>(N / kBlockN) * sizeof(float)};
  t[4] = {ks, nullptr, static_cast<size_t>(N / kBlockN) * sizeof(float)};
  t[5] = {vts, nullptr, static_cast<size_t>(d) * (N / 32)};
  t[6] = {nullptr, o, 2 * hb};
  t[7] = {nullptr, lse, static_cast<size_t>(N) * sizeof(float)};
  return 8;
}

// Largest sequence length accepted: keeps every position and mask limit of the
// kernels inside 32-bit integers.
constexpr long long kMaxSeq = 1ll << 30;

int validate_tensors(const void* q, const void* k, const void* v, const void* o, const void* lse, int B, int H,
                     int Nq, int Nk, int d, float scale) {
  if (!q || !k || !v || !o) return ATTN_ERR_NULL;
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return ATTN_ERR_DIMS;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED_HEADDIM;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_SCALE;
  const uintptr_t a = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                      reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
  if (a & 15u) return ATTN_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return ATTN_ERR_ALIGN;
  const long long BH = static_cast<long long>(B) * H;
  const long long qblocks = (static_cast<long long>(Nq) + kBlockM - 1) / kBlockM;
  if (Nq >= kMaxSeq || Nk >= kMaxSeq) return ATTN_ERR_OVERFLOW;
  if (BH > INT_MAX || BH * qblocks > INT_MAX) return ATTN_ERR_OVERFLOW;
  return ATTN_OK;
}

// Key-range splits a split-K/V launch actually uses for `requested` splits over
// num_kblocks key blocks: ranges of ceil(num_kblocks / requested) blocks, so
// there may be fewer ranges than requested (never more than key blocks).
struct SplitPlan {
  int blocks_per_split;
  int num_splits;
};
SplitPlan split_plan(int num_kblocks, int requested) {
  if (requested > num_kblocks) requested = num_kblocks;
  if (requested < 1) requested = 1;
  SplitPlan sp;
  sp.blocks_per_split = (num_kblocks + requested - 1) / requested;
  sp.num_splits = (num_kblocks + sp.blocks_per_split - 1) / sp.blocks_per_split;
  return sp;
}

// ---------------------------------------------------------------------------
// Unit order of unsplit causal launches.  Every candidate order is scored by the
// longest CTA's predicted time, walking the kernel's own schedule functions
// (unit_for_round, unit_info) with a unit costing max(n0, n1) + 2 K/V block
// periods (its two tiles advance together; 2 periods of prologue and epilogue).
// Candidates: zigzag, head-major and -- only for the BF16 instances that read
// their units from a table (table_cap > 0), where the order's arithmetic costs
// nothing at run time -- head groups whose K/V together stay under
// kPairOrderMaxKvBytes (a group of one head is always allowed), at most
// kMaxGroupCounts group counts.  A table instance takes every CTA's rounds
// from its table, so an order qualifies for it only when no CTA takes more
// rounds than the table holds; when none does, the launch goes to the table-less
// instance with zigzag or head-major order.  Ties keep the earlier candidate
// (zigzag, head-major, then the smaller groups: fewer bytes of K/V live in L2 at
// a time).  The choice is cached per shape.
// ---------------------------------------------------------------------------
constexpr double kUnitOverheadBlocks = 2.0;
constexpr int kMaxGroupCounts = 32;
constexpr long long kNoSearchRounds = 4 * kSchedEntries;  // zigzag's last round then costs < 0.5%
constexpr int kPairTailMinBlocks = 24;

int grid_for(const FwdParams& p, int num_sms) {
  // pair tail: CTA pairs, twice the units when they all fit in one split round
  if (p.pair_tail) {
    const long long g = 2ll * p.num_units < num_sms ? 2ll * p.num_units : num_sms;
    return static_cast<int>(g & ~1ll);
  }
  // work items dealt to CTAs: units, or combined heavy+light pairs under zigzag
  const int items = p.order == kOrderZigzag ? p.BH * ((p.num_pairs + 1) / 2) : p.num_units;
  return items < num_sms ? items : num_sms;
}

// Predicted makespan (K/V block periods) of p's order on num_sms SMs, and the
// most rounds (iterations, skipped ones included) a CTA takes.
double predicted_makespan(const FwdParams& p, int num_sms, int* max_rounds = nullptr) {
  const int G = grid_for(p, num_sms);
  double worst = 0.0;
  int rounds = 0;
  for (int c = 0; c < G; ++c) {
    double t = 0.0;
    int round = 0;
    for (;; ++round) {
      const int u = unit_for_round(round, p, G, c);
      if (u == kNoMoreUnits) break;
      if (u == kSkipRound) continue;
      const UnitInfo ui = unit_info(u, p, tail_role(round, p, G, c));
      t += (ui.n[1] > ui.n[0] ? ui.n[1] : ui.n[0]) + kUnitOverheadBlocks;
    }
    if (t > worst) worst = t;
    if (round > rounds) rounds = round;
  }
  if (max_rounds) *max_rounds = rounds;
  return worst;
}

using OrderKey = std::tuple<int, int, int, int, int, int, long long, int>;
struct OrderChoice {
  int order, group_heads, table;
};
std::map<OrderKey, OrderChoice> g_order_cache;
std::mutex g_order_mu;
int g_force_order = -1, g_force_group_heads = 0;  // attn_diag_force_fwd_order
std::atomic<bool> g_pair_tail_ok{true};            // attn_diag_set_pair_tail

// table_cap: rounds the unit table of the launch's kTable instance holds (0: the
// entry point has none)
void choose_order(FwdParams& p, int num_sms, long long kv_key_bytes, int table_cap, bool tail_untabled) {
  const bool table_ok = table_cap > 0;
  p.order = kOrderHeads;
  p.group_heads = p.BH;
  p.sched_table = 0;
  if (!p.causal || p.num_splits != 1) {
    // head-major: ceil(units / grid) rounds
    const int G = grid_for(p, num_sms);
    p.sched_table = table_ok && (p.num_units + G - 1) / G <= table_cap ? 1 : 0;
    // Pair tail (table launches, unsplit): when the last round holds at most one
    // unit per CTA pair, each of its units is split over a pair, so that round
    // takes half a unit's time (B1 H32 N4096: 512 units, 3.37 rounds of 152 CTAs
    // -> 3.5 unit times instead of 4).  The cluster launch and the exchange cost
    // ~12 us (measured: +4.7% at 32 key blocks of d = 128, -2% at 16), so only
    // units of at least kPairTailMinBlocks key blocks (twice that at d = 64, whose
    // blocks take about half the time) are split.
    const int min_kb = kv_key_bytes >= 4 * 128 ? kPairTailMinBlocks : 2 * kPairTailMinBlocks;
    if ((p.sched_table || tail_untabled) && p.num_splits == 1 && p.num_kblocks >= min_kb && g_pair_tail_ok &&
        num_sms >= 2) {
      FwdParams c = p;
      c.pair_tail = 1;
      const int Gp = grid_for(c, num_sms);
      const int full = p.num_units / Gp, rem = p.num_units - full * Gp;
      if (rem > 0 && 2 * rem <= Gp && (!p.sched_table || full + 1 <= table_cap)) p.pair_tail = 1;
    }
    return;
  }
  int force_order, force_hg;
  {
    std::lock_guard<std::mutex> lk(g_order_mu);
    force_order = g_force_order;
    force_hg = g_force_group_heads;
  }
  if (force_order >= 0) {
    p.order = force_order;
    p.group_heads = force_hg > 0 && force_hg < p.BH ? force_hg : p.BH;
    int rounds = 0;
    if (table_ok) predicted_makespan(p, num_sms, &rounds);
    p.sched_table = table_ok && rounds <= table_cap ? 1 : 0;
    return;
  }
  if (p.num_units > kNoSearchRounds * num_sms) {  // many rounds: the tail costs little, skip the search
    p.order = kOrderZigzag;
    return;
  }
  const OrderKey key{p.BH, p.Nq, p.Nk, p.q_offset, p.k_offset, num_sms, kv_key_bytes, table_cap};
  {
    std::lock_guard<std::mutex> lk(g_order_mu);
    const auto it = g_order_cache.find(key);
    if (it != g_order_cache.end()) {
      p.order = it->second.order;
      p.group_heads = it->second.group_heads;
      p.sched_table = it->second.table;
      return;
    }
  }
  FwdParams c = p;
  // best order with the table (every CTA within table_cap rounds) and without
  OrderChoice best_tab{-1, p.BH, 1}, best_inl{-1, p.BH, 0};
  double t_tab = 0.0, t_inl = 0.0;
  auto consider = [&](int order, int hg) {
    c.order = order;
    c.group_heads = hg;
    int rounds = 0;
    const double t = predicted_makespan(c, num_sms, &rounds);
    if (order != kOrderGroups && (best_inl.order < 0 || t < t_inl * (1.0 - 1e-3))) {
      best_inl = {order, hg, 0};
      t_inl = t;
    }
    if (table_ok && rounds <= table_cap && (best_tab.order < 0 || t < t_tab * (1.0 - 1e-3))) {
      best_tab = {order, hg, 1};
      t_tab = t;
    }
  };
  consider(kOrderZigzag, p.BH);
  consider(kOrderHeads, p.BH);
  if (table_ok) {
    const long long head_kv = static_cast<long long>(p.Nk) * kv_key_bytes;
    int last_hg = 0;
    for (int groups = p.BH < kMaxGroupCounts ? p.BH : kMaxGroupCounts; groups >= 1; --groups) {
      const int hg = (p.BH + groups - 1) / groups;  // increasing with fewer groups
      if (hg == last_hg) continue;
      last_hg = hg;
      if (hg > 1 && hg * head_kv > kPairOrderMaxKvBytes) break;
      consider(kOrderGroups, hg);
    }
  }
  const OrderChoice pick = best_tab.order >= 0 ? best_tab : best_inl;
  p.order = pick.order;
  p.group_heads = pick.group_heads;
  p.sched_table = pick.table;
  std::lock_guard<std::mutex> lk(g_order_mu);
  if (g_order_cache.size() >= 4096) g_order_cache.clear();
  g_order_cache[key] = pick;
}

// kv_key_bytes: bytes of one key's K and V rows together (sizes the L2 cap of the
// unit order)
// table_ok: the launch may go to a kTable instance (the BF16 final-output entry
// points); the table holds kSchedEntries rounds, kSchedEntriesTma in the
// instances with the O staging buffers (non-causal)
// tail_untabled: the launch may split its last round over CTA pairs without the
// unit table (the FP8 entry points, whose instances compute their units)
void fill_params(FwdParams& p, int BH, int Nq, int Nk, int causal, int q_offset, int k_offset, int num_splits,
                 float scale, int num_sms, long long kv_key_bytes, bool table_ok, bool tail_untabled = false) {
  std::memset(&p, 0, sizeof(p));
  p.BH = BH;
  p.Nq = Nq;
  p.Nk = Nk;
  p.q_offset = q_offset;
  p.k_offset = k_offset;
  p.num_kblocks = (Nk + kBlockN - 1) / kBlockN;
  p.num_pairs = (Nq + kTilesPerUnit * kBlockM - 1) / (kTilesPerUnit * kBlockM);
  const SplitPlan sp = split_plan(p.num_kblocks, num_splits);
  p.blocks_per_split = sp.blocks_per_split;
  p.num_splits = sp.num_splits;
  p.num_units = BH * p.num_pairs * p.num_splits;
  p.causal = causal ? 1 : 0;
  choose_order(p, num_sms, kv_key_bytes, !table_ok ? 0 : (causal ? kSchedEntries : kSchedEntriesTma),
               tail_untabled);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = g_timeout_ns;
}

// mo: tensor map of the bf16 output O (read only by the kTmaO instances)
template <int D, int NK, int NV, bool kFp8, bool kPartial, bool kFp4 = false, bool kTmaO = false,
          bool kTable = false, bool kPairTail = false>
int launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mo,
           const FwdParams& p, int dev, void* stream) {
  // the host's own bookkeeping: the instance matches the schedule
  if (static_cast<bool>(p.sched_table) != kTable || static_cast<bool>(p.pair_tail) != kPairTail)
    return ATTN_ERR_LAUNCH;
  const int grid = grid_for(p, g_dev[dev].num_sms);
  constexpr size_t smem = SmemPlan<D, NK, NV, kFp8, kFp4, kTmaO, kTable>::kBytes;
  FwdParams pk = p;
  pk.o_align32 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;  // the API requires 16 only
  auto kernel = attn_fwd_kernel<D, NK, NV, kFp8, kPartial, kFp4, kTmaO, kTable, kPairTail>;
  if constexpr (kPairTail) {
    // clusters of two CTAs (the pairs of the split last round)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kNumThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, mq, mk, mv, mo, pk) != cudaSuccess) return ATTN_ERR_LAUNCH;
  } else {
    kernel<<<grid, kNumThreads, smem, static_cast<cudaStream_t>(stream)>>>(mq, mk, mv, mo, pk);
  }
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

// BF16 launch over q [BH, Nq, d], k/v [BH, Nk, d] with the parameters in p;
// `partial` selects the per-split fp32 output.
int launch_bf16(const void* q, const void* k, const void* v, int d, bool partial, FwdParams& p, int dev,
                void* stream) {
  int rc;
  CUtensorMap mq, mk, mv;
  if ((rc = make_map(&mq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, p.Nq, p.BH, 64)) != ATTN_OK) return rc;
  if ((rc = make_map(&mk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, p.Nk, p.BH, 64)) != ATTN_OK) return rc;
  if ((rc = make_map(&mv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, p.Nk, p.BH, 64)) != ATTN_OK) return rc;
  if (partial) {
    if (d == 64) return launch<ATTN_BF16_D64, true>(mq, mk, mv, mq, p, dev, stream);
    return launch<ATTN_BF16_D128, true>(mq, mk, mv, mq, p, dev, stream);
  }
  // Non-causal launches store O through shared-memory staging and TMA (+2-5% on
  // B4 H16 N2048 d128, B16 H16 N4096 d64 and B1 H32 N4096 d128, measured A/B
  // against row-per-thread stores); causal ones keep the row stores (the staging
  // buffer cost 3% on B4 H16 N2048 d128 causal, whose units are short).
  if (p.causal) {
    if (p.sched_table) {
      if (d == 64) return launch<ATTN_BF16_D64, false, false, false, true>(mq, mk, mv, mq, p, dev, stream);
      return launch<ATTN_BF16_D128, false, false, false, true>(mq, mk, mv, mq, p, dev, stream);
    }
    if (d == 64) return launch<ATTN_BF16_D64, false>(mq, mk, mv, mq, p, dev, stream);
    return launch<ATTN_BF16_D128, false>(mq, mk, mv, mq, p, dev, stream);
  }
  CUtensorMap mo;
  if ((rc = make_map(&mo, p.o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, p.Nq, p.BH, 64)) != ATTN_OK) return rc;
  if (p.pair_tail) {
    if (d == 64) return launch<ATTN_BF16_D64, false, false, true, true, true>(mq, mk, mv, mo, p, dev, stream);
    return launch<ATTN_BF16_D128, false, false, true, true, true>(mq, mk, mv, mo, p, dev, stream);
  }
  if (p.sched_table) {
    if (d == 64) return launch<ATTN_BF16_D64, false, false, true, true>(mq, mk, mv, mo, p, dev, stream);
    return launch<ATTN_BF16_D128, false, false, true, true>(mq, mk, mv, mo, p, dev, stream);
  }
  if (d == 64) return launch<ATTN_BF16_D64, false, false, true>(mq, mk, mv, mo, p, dev, stream);
  return launch<ATTN_BF16_D128, false, false, true>(mq, mk, mv, mo, p, dev, stream);
}

int launch_merge(const float* const* o_parts, const float* const* lse_parts, int S, void* out, float* lse_out,
                 int out_fp32, long long rows, int d, int dev, void* stream) {
  MergeParams mp;
  std::memset(&mp, 0, sizeof(mp));
  for (int s = 0; s < S; ++s) {
    mp.o[s] = o_parts[s];
    mp.lse[s] = lse_parts[s];
  }
  mp.S = S;
  mp.out = out;
  mp.lse_out = lse_out;
  mp.out_fp32 = out_fp32;
  mp.rows = rows;
  const long long warps_needed = rows;
  long long blocks = (warps_needed + 7) / 8;  // 8 warps per 256-thread block
  const long long cap = static_cast<long long>(g_dev[dev].num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (d == 64) attn_merge_kernel<64><<<static_cast<int>(blocks), 256, 0, st>>>(mp);
  else attn_merge_kernel<128><<<static_cast<int>(blocks), 256, 0, st>>>(mp);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

size_t splitkv_workspace_bytes(long long BH, long long Nq, long long d, long long S) {
  const long long rows = BH * Nq;
  // O partials, then lse partials (each partial's O block stays 16-byte aligned)
  return static_cast<size_t>(S * rows * d * 4 + S * rows * 4);
}

}  // namespace

namespace {
template <int D, int RA, int RB>
int launch_bwd(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdo,
               const BwdParams& bp, int dev, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long rows = static_cast<long long>(bp.BH) * bp.Npad;
  long long pblocks = (rows + 7) / 8;
  const long long cap = static_cast<long long>(g_dev[dev].num_sms) * 8;
  if (pblocks > cap) pblocks = cap;
  attn_bwd_prep_kernel<D><<<static_cast<int>(pblocks), 256, 0, st>>>(bp);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  // CTAs: units, or block pairs under the zigzag order
  const int items = bp.order == kBwdOrderZigzag ? bp.BH * ((bp.num_blocks + 1) / 2) : bp.num_units;
  const int grid = items < g_dev[dev].num_sms ? items : g_dev[dev].num_sms;
  const size_t smem = BwdSmem<D, RA, RB>::kBytes;
  attn_bwd_dq_kernel<D, RA, RB><<<grid, kBwdThreads, smem, st>>>(mq, mk, mv, mdo, bp);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  attn_bwd_dkdv_kernel<D, RA, RB><<<grid, kDkdvThreads, smem, st>>>(mq, mk, mv, mdo, bp);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}
// The pipeline of the host-buffer entry points: chunks of whole heads through two
// workspace slots; per chunk the inputs are copied in on s_in, `launch(h0, hn,
// dev)` runs the kernel on the caller's stream with dev[i] = the slot's region of
// tensor i, and the outputs are copied back on s_out.  Null host pointers (an
// optional LSE) are skipped.
template <class Launch>
int host_pipeline(const HostTensor* t, int nt, const HostChunking& hcfg, long long BH, void* workspace, int dev,
                  void* stream, Launch launch) {
  HostPipe& hp = g_pipe[dev];
  std::lock_guard<std::mutex> lock(hp.mu);
  int rc;
  if ((rc = pipe_setup(hp)) != ATTN_OK) return rc;
  cudaStream_t sc = static_cast<cudaStream_t>(stream);
  bool ok = true;
  auto ck = [&ok](cudaError_t e) { ok = ok && e == cudaSuccess; };
  // the copies wait for earlier work on the caller's stream (it may still use the workspace)
  ck(cudaEventRecord(hp.entry, sc));
  ck(cudaStreamWaitEvent(hp.s_in, hp.entry, 0));
  ck(cudaStreamWaitEvent(hp.s_out, hp.entry, 0));
  for (int c = 0; c < hcfg.chunks && ok; ++c) {
    const int slot = c % kHostSlots;
    const long long h0 = static_cast<long long>(c) * hcfg.heads;
    const int hn = static_cast<int>(BH - h0 < hcfg.heads ? BH - h0 : hcfg.heads);
    uint8_t* reg[kHostMaxTensors];
    uint8_t* base = static_cast<uint8_t*>(workspace) + slot * hcfg.slot_bytes;
    for (int i = 0; i < nt; ++i) {
      reg[i] = base;
      base += hcfg.region[i];
    }
    // copy in, once the kernel two chunks back is done with this slot's inputs
    if (c >= kHostSlots) ck(cudaStreamWaitEvent(hp.s_in, hp.comp_done[slot], 0));
    for (int i = 0; i < nt; ++i)
      if (t[i].in)
        ck(cudaMemcpyAsync(reg[i], static_cast<const uint8_t*>(t[i].in) + h0 * t[i].per_head, hn * t[i].per_head,
                           cudaMemcpyHostToDevice, hp.s_in));
    ck(cudaEventRecord(hp.in_done[slot], hp.s_in));
    // the kernel, once the inputs are in and the copy-out two chunks back has read the outputs
    ck(cudaStreamWaitEvent(sc, hp.in_done[slot], 0));
    if (c >= kHostSlots) ck(cudaStreamWaitEvent(sc, hp.out_done[slot], 0));
    if (!ok) break;
    if ((rc = launch(h0, hn, reg)) != ATTN_OK) return rc;
    ck(cudaEventRecord(hp.comp_done[slot], sc));
    // copy out
    ck(cudaStreamWaitEvent(hp.s_out, hp.comp_done[slot], 0));
    for (int i = 0; i < nt; ++i)
      if (t[i].out)
        ck(cudaMemcpyAsync(static_cast<uint8_t*>(t[i].out) + h0 * t[i].per_head, reg[i], hn * t[i].per_head,
                           cudaMemcpyDeviceToHost, hp.s_out));
    ck(cudaEventRecord(hp.out_done[slot], hp.s_out));
  }
  // work queued on the caller's stream after this call sees the outputs in host memory
  ck(cudaEventRecord(hp.last, hp.s_out));
  ck(cudaStreamWaitEvent(sc, hp.last, 0));
  return ok ? ATTN_OK : ATTN_ERR_CUDA;
}

int launch_fp8(const void* q8, const void* k8, const void* v8, const float* q_scale, const float* k_scale,
               const float* v_scale, void* o, float* lse, int BH, int N, int d, int causal, float scale, int dev,
               void* stream);
int launch_fp4p(const void* q8, const void* k8, const void* vt4, const float* q_scale, const float* k_scale,
                const uint8_t* vt_scale, void* o, float* lse, int BH, int N, int d, int causal, float scale, int dev,
                void* stream);

}  // namespace

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
             int causal, float scale, int dtype, void* stream) {
  int rc = validate_tensors(q, k, v, o, lse, B, H, N, N, d, scale);
  if (rc != ATTN_OK) return rc;
  if (dtype != ATTN_BF16) return ATTN_ERR_DTYPE;
  int dev = 0;
  if ((rc = device_setup(&dev)) != ATTN_OK) return rc;
  FwdParams p;
  fill_params(p, B * H, N, N, causal, 0, 0, 1, scale, g_dev[dev].num_sms, 4ll * d, true);
  p.err = g_dev[dev].err_ptr;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  return launch_bf16(q, k, v, d, false, p, dev, stream);
}

size_t attn_fwd_host_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return 0;
  HostTensor t[kHostMaxTensors];
  const int nt = bf16_host_tensors(t, nullptr, nullptr, nullptr, nullptr, nullptr, N, d);
  return kHostSlots * host_chunking(B, H, t, nt).slot_bytes;
}

int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                  int causal, float scale, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = validate_tensors(q, k, v, o, lse, B, H, N, N, d, scale);
  if (rc != ATTN_OK) return rc;
  if (!workspace) return ATTN_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_ALIGN;
  HostTensor t[kHostMaxTensors];
  const int nt = bf16_host_tensors(t, q, k, v, o, lse, N, d);
  const HostChunking hcfg = host_chunking(B, H, t, nt);
  if (workspace_bytes < kHostSlots * hcfg.slot_bytes) return ATTN_ERR_WORKSPACE;
  int dev = 0;
  if ((rc = device_setup(&dev)) != ATTN_OK) return rc;
  return host_pipeline(t, nt, hcfg, static_cast<long long>(B) * H, workspace, dev, stream,
                       [&](long long, int hn, uint8_t* const* reg) {
                         FwdParams p;
                         fill_params(p, hn, N, N, causal, 0, 0, 1, scale, g_dev[dev].num_sms, 4ll * d, true);
                         p.err = g_dev[dev].err_ptr;
                         p.o = reinterpret_cast<__nv_bfloat16*>(reg[3]);
                         p.lse = lse ? reinterpret_cast<float*>(reg[4]) : nullptr;
                         return launch_bf16(reg[0], reg[1], reg[2], d, false, p, dev, stream);
                       });
}

size_t attn_fwd_fp8_host_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d != 128) return 0;
  HostTensor t[kHostMaxTensors];
  const int nt = fp8_host_tensors(t, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, N, d);
  return kHostSlots * host_chunking(B, H, t, nt).slot_bytes;
}

int attn_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* q_scale, const float* k_scale,
                 const float* v_scale, void* o, float* lse, int B, int H, int N, int d, int causal, float scale,
                 void* stream) {
  int rc = validate_tensors(q8, k8, v8, o, lse, B, H, N, N, d, scale);
  if (rc != ATTN_OK) return rc;
  if (d != 128) return ATTN_ERR_UNSUPPORTED_HEADDIM;
  if (!q_scale || !k_scale || !v_scale) return ATTN_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(q_scale) | reinterpret_cast<uintptr_t>(k_scale) |
       reinterpret_cast<uintptr_t>(v_scale)) & 3u)
    return ATTN_ERR_ALIGN;
  int dev = 0;
  if ((rc = device_setup(&dev)) != ATTN_OK) return rc;
  return launch_fp8(q8, k8, v8, q_scale, k_scale, v_scale, o, lse, B * H, N, d, causal, scale, dev, stream);
}

int attn_fwd_fp8_host(const void* q8, const void* k8, const void* v8, const float* q_scale, const float* k_scale,
                      const float* v_scale, void* o, float* lse, int B, int H, int N, int d, int causal, float scale,
                      void* workspace, size_t workspace_bytes, void* stream) {
  int rc = validate_tensors(q8, k8, v8, o, lse, B, H, N, N, d, scale);
  if (rc != ATTN_OK) return rc;
  if (d != 128) return ATTN_ERR_UNSUPPORTED_HEADDIM;
  if (!q_scale || !k_scale || !v_scale || !workspace) return ATTN_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_ALIGN;
  HostTensor t[kHostMaxTensors];
  const int nt = fp8_host_tensors(t, q8, k8, v8, q_scale, k_scale, v_scale, o, lse, N, d);
  const HostChunking hcfg = host_chunking(B, H, t, nt);
  if (workspace_bytes < kHostSlots * hcfg.slot_bytes) return ATTN_ERR_WORKSPACE;
  int dev = 0;
  if ((rc = device_setup(&dev)) != ATTN_OK) return rc;
  return host_pipeline(t, nt, hcfg, static_cast<long long>(B) * H, workspace, dev, stream,
                       [&](long long, int hn, uint8_t* const* reg) {
                         return launch_fp8(reg[0], reg[1], reg[2], reinterpret_cast<const float*>(reg[3]),
                                           reinterpret_cast<const float*>(reg[4]),
                                           reinterpret_cast<const float*>(reg[5]), reg[6],
                                           lse ? reinterpret_cast<float*>(reg[7]) : nullptr, hn, N, d, causal,
                                           scale, dev, stream);
                       });
}

}  // extern "C"

namespace {
// The FP8 forward over BH heads of device tensors (arguments already checked).
int launch_fp8(const void* q8, const void* k8, const void* v8, const float* q_scale, const float* k_scale,
               const float* v_scale, void* o, float* lse, int BH, int N, int d, int causal, float scale, int dev,
               void* stream) {
  int rc;
  CUtensorMap mq, mk, mv;
  if ((rc = make_map(&mq, q8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, d, N, BH, 128)) != ATTN_OK) return rc;
  if ((rc = make_map(&mk, k8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, d, N, BH, 128)) != ATTN_OK) return rc;
  if ((rc = make_map(&mv, v8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, d, N, BH, 128)) != ATTN_OK) return rc;
  FwdParams p;
  fill_params(p, BH, N, N, causal, 0, 0, 1, scale, g_dev[dev].num_sms, 2ll * d, false, true);
  p.err = g_dev[dev].err_ptr;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.q_scale = q_scale;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  if (p.pair_tail) return launch<ATTN_FP8_D128, false, false, false, false, true>(mq, mk, mv, mq, p, dev, stream);
  return launch<ATTN_FP8_D128, false>(mq, mk, mv, mq, p, dev, stream);
}
}  // namespace

extern "C" {

int attn_fwd_fp4p(const void* q8, const void* k8, const void* vt4, const float* q_scale, const float* k_scale,
                  const uint8_t* vt_scale, void* o, float* lse, int B, int H, int N, int d, int causal, float scale,
                  void* stream) {
  int rc = validate_tensors(q8, k8, vt4, o, lse, B, H, N, N, d, scale);
  if (rc != ATTN_OK) return rc;
  if (d != 128) return ATTN_ERR_UNSUPPORTED_HEADDIM;
  if (N % kBlockN != 0) return ATTN_ERR_DIMS;
  // the kernel indexes the scale words of V^T with 32-bit integers
  if (static_cast<long long>(B) * H * d * (N / kBlockN) >= (1ll << 32)) return ATTN_ERR_OVERFLOW;
  if (!q_scale || !k_scale || !vt_scale) return ATTN_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(q_scale) | reinterpret_cast<uintptr_t>(k_scale) |
       reinterpret_cast<uintptr_t>(vt_scale)) & 3u)
    return ATTN_ERR_ALIGN;
  int dev = 0;
  if ((rc = device_setup(&dev)) != ATTN_OK) return rc;
  return launch_fp4p(q8, k8, vt4, q_scale, k_scale, vt_scale, o, lse, B * H, N, d, causal, scale, dev, stream);
}

int attn_fwd_fp4p_host(const void* q8, const void* k8, const void* vt4, const float* q_scale, const float* k_scale,
                       const uint8_t* vt_scale, void* o, float* lse, int B, int H, int N, int d, int causal,
                       float scale, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = validate_tensors(q8, k8, vt4, o, lse, B, H, N, N, d, scale);
  if (rc != ATTN_OK) return rc;
  if (d != 128) return ATTN_ERR_UNSUPPORTED_HEADDIM;
  if (N % kBlockN != 0) return ATTN_ERR_DIMS;
  // the kernel indexes the scale words of V^T with 32-bit integers (per chunk; all heads bound it)
  if (static_cast<long long>(B) * H * d * (N / kBlockN) >= (1ll << 32)) return ATTN_ERR_OVERFLOW;
  if (!q_scale || !k_scale || !vt_scale || !workspace) return ATTN_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_ALIGN;
  HostTensor t[kHostMaxTensors];
  const int nt = fp4p_host_tensors(t, q8, k8, vt4, q_scale, k_scale, vt_scale, o, lse, N, d);
  const HostChunking hcfg = host_chunking(B, H, t, nt);
  if (workspace_bytes < kHostSlots * hcfg.slot_bytes) return ATTN_ERR_WORKSPACE;
  int dev = 0;
  if ((rc = device_setup(&dev)) != ATTN_OK) return rc;
  return host_pipeline(t, nt, hcfg, static_cast<long long>(B) * H, workspace, dev, stream,
                       [&](long long, int hn, uint8_t* const* reg) {
                         return launch_fp4p(reg[0], reg[1], reg[2], reinterpret_cast<const float*>(reg[3]),
                                            reinterpret_cast<const float*>(reg[4]), reg[5], reg[6],
                                            lse ? reinterpret_cast<float*>(reg[7]) : nullptr, hn, N, d, causal,
                                            scale, dev, stream);
                       });
}

size_t attn_fwd_fp4p_host_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d != 128 || N % kBlockN != 0) return 0;
  HostTensor t[kHostMaxTensors];
  const int nt = fp4p_host_tensors(t, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, N, d);
  return kHostSlots * host_chunking(B, H, t, nt).slot_bytes;
}

}  // extern "C"

namespace {
// The Direct-P FP4 forward over BH heads of device tensors (arguments already checked).
int launch_fp4p(const void* q8, const void* k8, const void* vt4, const float* q_scale, const float* k_scale,
                const uint8_t* vt_scale, void* o, float* lse, int BH, int N, int d, int causal, float scale, int dev,
                void* stream) {
  int rc;
  CUtensorMap mq, mk, mv;
  if ((rc = make_map(&mq, q8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, d, N, BH, 128)) != ATTN_OK) return rc;
  if ((rc = make_map(&mk, k8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, d, N, BH, 128)) != ATTN_OK) return rc;
  if ((rc = make_map_vt4(&mv, vt4, d, N, BH)) != ATTN_OK) return rc;
  FwdParams p;
  fill_params(p, BH, N, N, causal, 0, 0, 1, scale, g_dev[dev].num_sms, 2ll * d, false);
  p.err = g_dev[dev].err_ptr;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.q_scale = q_scale;
  p.k_scale = k_scale;
  p.v_scale = reinterpret_cast<const float*>(vt_scale);  // E8M0 words, read as such by the FP4 path
  return launch<ATTN_FP4_D128, false, true>(mq, mk, mv, mq, p, dev, stream);
}
}  // namespace

extern "C" {

int attn_fwd_partial(const void* q, const void* k, const void* v, float* o_part, float* lse_part, int B, int H,
                     int Nq, int Nk, int d, int causal, int q_offset, int k_offset, float scale, void* stream) {
  int rc = validate_tensors(q, k, v, o_part, lse_part, B, H, Nq, Nk, d, scale);
  if (rc != ATTN_OK) return rc;
  if (!lse_part) return ATTN_ERR_NULL;
  if (q_offset < 0 || k_offset < 0 || q_offset >= kMaxSeq || k_offset >= kMaxSeq) return ATTN_ERR_DIMS;
  int dev = 0;
  if ((rc = device_setup(&dev)) != ATTN_OK) return rc;
  FwdParams p;
  fill_params(p, B * H, Nq, Nk, causal, q_offset, k_offset, 1, scale, g_dev[dev].num_sms, 4ll * d, false);
  p.err = g_dev[dev].err_ptr;
  p.o_part = o_part;
  p.lse_part = lse_part;
  return launch_bf16(q, k, v, d, true, p, dev, stream);
}

int attn_merge(const float* const* o_parts, const float* const* lse_parts, int num_parts, void* o, float* lse,
               int out_fp32, int B, int H, int N, int d, void* stream) {
  if (!o_parts || !lse_parts || !o) return ATTN_ERR_NULL;
  if (num_parts < 1 || num_parts > kMaxMergeParts || B < 1 || H < 1 || N < 1) return ATTN_ERR_DIMS;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED_HEADDIM;
  uintptr_t a = reinterpret_cast<uintptr_t>(o);
  for (int s = 0; s < num_parts; ++s) {
    if (!o_parts[s] || !lse_parts[s]) return ATTN_ERR_NULL;
    a |= reinterpret_cast<uintptr_t>(o_parts[s]);
    if (reinterpret_cast<uintptr_t>(lse_parts[s]) & 3u) return ATTN_ERR_ALIGN;
  }
  if ((a & 15u) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_ALIGN;
  if (static_cast<long long>(B) * H * N > (1ll << 40)) return ATTN_ERR_OVERFLOW;
  int dev = 0;
  int rc = device_setup(&dev);
  if (rc != ATTN_OK) return rc;
  return launch_merge(o_parts, lse_parts, num_parts, o, lse, out_fp32 ? 1 : 0,
                      static_cast<long long>(B) * H * N, d, dev, stream);
}

size_t attn_splitkv_workspace_bytes(int B, int H, int Nq, int d, int num_splits) {
  if (B < 1 || H < 1 || Nq < 1 || (d != 64 && d != 128) || num_splits < 1 || num_splits > kMaxMergeParts) return 0;
  return splitkv_workspace_bytes(static_cast<long long>(B) * H, Nq, d, num_splits);
}

int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                     int Nk, int d, int causal, float scale, int num_splits, void* workspace,
                     size_t workspace_bytes, void* stream) {
  int rc = validate_tensors(q, k, v, o, lse, B, H, Nq, Nk, d, scale);
  if (rc != ATTN_OK) return rc;
  if (num_splits < 1 || num_splits > kMaxMergeParts) return ATTN_ERR_DIMS;
  if (causal && Nq > Nk) return ATTN_ERR_DIMS;
  if (!workspace) return ATTN_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(workspace) & 15u) return ATTN_ERR_ALIGN;
  int dev = 0;
  if ((rc = device_setup(&dev)) != ATTN_OK) return rc;
  const int BH = B * H;
  FwdParams p;
  // causal: the queries are the last Nq positions of the Nk keys
  fill_params(p, BH, Nq, Nk, causal, Nk - Nq, 0, num_splits, scale, g_dev[dev].num_sms, 4ll * d, false);
  p.err = g_dev[dev].err_ptr;
  const long long S = p.num_splits;
  if (workspace_bytes < splitkv_workspace_bytes(BH, Nq, d, S)) return ATTN_ERR_WORKSPACE;
  const long long rows = static_cast<long long>(BH) * Nq;
  float* o_part = static_cast<float*>(workspace);
  float* lse_part = o_part + S * rows * d;
  p.o_part = o_part;
  p.lse_part = lse_part;
  if ((rc = launch_bf16(q, k, v, d, true, p, dev, stream)) != ATTN_OK) return rc;
  const float* op[kMaxMergeParts];
  const float* lp[kMaxMergeParts];
  for (int s = 0; s < S; ++s) {
    op[s] = o_part + s * rows * d;
    lp[s] = lse_part + s * rows;
  }
  return launch_merge(op, lp, static_cast<int>(S), o, lse, 0, rows, d, dev, stream);
}

size_t attn_bwd_workspace_bytes(int B, int H, int N) {
  if (B < 1 || H < 1 || N < 1) return 0;
  // two float arrays [B*H][N rounded up to 128]: -lse log2e and -scale D_i
  const size_t npad = (static_cast<size_t>(N) + kBlockM - 1) / kBlockM * kBlockM;
  return 2 * static_cast<size_t>(B) * H * npad * sizeof(float);
}


int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
             void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale, void* workspace,
             size_t workspace_bytes, void* stream) {
  int rc = validate_tensors(q, k, v, o, nullptr, B, H, N, N, d, scale);
  if (rc != ATTN_OK) return rc;
  if (!dout || !lse || !dq || !dk || !dv || !workspace) return ATTN_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(dq) | reinterpret_cast<uintptr_t>(dk) |
       reinterpret_cast<uintptr_t>(dv)) & 15u)
    return ATTN_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return ATTN_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(workspace) & 15u) return ATTN_ERR_ALIGN;
  if (workspace_bytes < attn_bwd_workspace_bytes(B, H, N)) return ATTN_ERR_WORKSPACE;
  int dev = 0;
  if ((rc = device_setup(&dev)) != ATTN_OK) return rc;
  const int BH = B * H;
  CUtensorMap mq, mk, mv, mdo;
  if ((rc = make_map(&mq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, N, BH, 64)) != ATTN_OK) return rc;
  if ((rc = make_map(&mk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, N, BH, 64)) != ATTN_OK) return rc;
  if ((rc = make_map(&mv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, N, BH, 64)) != ATTN_OK) return rc;
  if ((rc = make_map(&mdo, dout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, N, BH, 64)) != ATTN_OK) return rc;
  BwdParams bp;
  std::memset(&bp, 0, sizeof(bp));
  bp.o = static_cast<const __nv_bfloat16*>(o);
  bp.dout = static_cast<const __nv_bfloat16*>(dout);
  bp.lse = lse;
  bp.num_blocks = (N + kBlockN - 1) / kBlockN;
  bp.Npad = bp.num_blocks * kBlockN;
  bp.nlse2 = static_cast<float*>(workspace);
  bp.nds = bp.nlse2 + static_cast<size_t>(B) * H * bp.Npad;
  bp.dq = static_cast<__nv_bfloat16*>(dq);
  bp.dk = static_cast<__nv_bfloat16*>(dk);
  bp.dv = static_cast<__nv_bfloat16*>(dv);
  bp.BH = BH;
  bp.N = N;
  bp.num_units = BH * bp.num_blocks;
  bp.causal = causal ? 1 : 0;
  bp.order = kBwdOrderHeads;
  if (causal) {
    // both passes stream two tensors of d bf16 per key per head (K, V or Q, dO)
    const long long streamed = static_cast<long long>(BH) * bp.Npad * 4ll * d;
    if (streamed <= kPairOrderMaxKvBytes) bp.order = kBwdOrderBlocks;
    else if (static_cast<long long>(BH) * ((bp.num_blocks + 1) / 2) >= 4ll * g_dev[dev].num_sms)
      bp.order = kBwdOrderZigzag;
  }
  bp.scale = scale;
  bp.scale_log2 = scale * 1.4426950408889634f;
  bp.timeout_ns = g_timeout_ns;
  bp.err = g_dev[dev].err_ptr;
  if (d == 64) return launch_bwd<ATTN_BWD_D64>(mq, mk, mv, mdo, bp, dev, stream);
  return launch_bwd<ATTN_BWD_D128>(mq, mk, mv, mdo, bp, dev, stream);
}

int attn_bwd_host(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                  void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale, void* workspace,
                  size_t workspace_bytes, void* stream) {
  int rc = validate_tensors(q, k, v, o, nullptr, B, H, N, N, d, scale);
  if (rc != ATTN_OK) return rc;
  if (!dout || !lse || !dq || !dk || !dv || !workspace) return ATTN_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_ALIGN;
  HostTensor t[kHostMaxTensors];
  const int nt = bwd_host_tensors(t, q, k, v, o, dout, lse, dq, dk, dv, N, d);
  const HostChunking hcfg = host_chunking(B, H, t, nt);
  if (workspace_bytes < kHostSlots * hcfg.slot_bytes) return ATTN_ERR_WORKSPACE;
  int dev = 0;
  if ((rc = device_setup(&dev)) != ATTN_OK) return rc;
  return host_pipeline(t, nt, hcfg, static_cast<long long>(B) * H, workspace, dev, stream,
                       [&](long long, int hn, uint8_t* const* reg) {
                         return attn_bwd(reg[0], reg[1], reg[2], reg[3], reg[4], reinterpret_cast<const float*>(reg[5]),
                                         reg[6], reg[7], reg[8], 1, hn, N, d, causal, scale, reg[9],
                                         hcfg.region[9], stream);
                       });
}

size_t attn_bwd_host_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return 0;
  HostTensor t[kHostMaxTensors];
  const int nt = bwd_host_tensors(t, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, N,
                                  d);
  return kHostSlots * host_chunking(B, H, t, nt).slot_bytes;
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_NULL: return "ATTN_ERR_NULL: a required pointer is NULL";
    case ATTN_ERR_DIMS: return "ATTN_ERR_DIMS: a size or count is out of range (B, H, N must be >= 1)";
    case ATTN_ERR_UNSUPPORTED_HEADDIM: return "ATTN_ERR_UNSUPPORTED_HEADDIM: d must be 64 or 128";
    case ATTN_ERR_DTYPE: return "ATTN_ERR_DTYPE: unknown dtype";
    case ATTN_ERR_ALIGN: return "ATTN_ERR_ALIGN: tensors must be 16-byte aligned (lse/scales 4-byte)";
    case ATTN_ERR_OVERFLOW: return "ATTN_ERR_OVERFLOW: sizes exceed 32-bit work indexing or TMA limits";
    case ATTN_ERR_LAUNCH: return "ATTN_ERR_LAUNCH: kernel launch failed";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT: a bounded in-kernel wait ran out";
    case ATTN_ERR_ARCH: return "ATTN_ERR_ARCH: the current device is not sm_103";
    case ATTN_ERR_SCALE: return "ATTN_ERR_SCALE: scale must be finite and > 0";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA: a CUDA call failed (no device?)";
    case ATTN_ERR_SCRATCH: return "ATTN_ERR_SCRATCH: the problem needs more than the library's fixed scratch";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE: the workspace is smaller than its *_workspace_bytes()";
    default: return "unknown attn_status";
  }
}

int attn_check_device_errors(void* stream, int* where_out) {
  int dev = 0;
  int rc = device_setup(&dev);
  if (rc != ATTN_OK) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  int word = 0;
  const int zero = 0;
  if (cudaMemcpyFromSymbol(&word, g_attn_err, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_attn_err, &zero, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
  if (where_out) *where_out = word >> 8;
  return (word & 0xff) == kDevErrTimeout ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

int attn_set_wait_timeout_ns(unsigned long long ns) {
  if (ns < 1000ull) return ATTN_ERR_DIMS;
  g_timeout_ns = ns;
  return ATTN_OK;
}

}  // extern "C"

namespace {
// One CTA waits on an mbarrier that nothing ever arrives at; the bounded wait
// must give up, record the timeout and let the kernel exit normally.
__global__ void wait_selftest_kernel(unsigned long long timeout_ns, int* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_word;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_word = 0;
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait(smem_u32(&bar), 0, &abort_word, timeout_ns, err, 99);
}
}  // namespace

extern "C" int attn_diag_set_pair_tail(int enable) {
  g_pair_tail_ok = enable != 0;
  return ATTN_OK;
}

extern "C" int attn_diag_force_fwd_order(int order, int group_heads) {
  if (order < -1 || order > kOrderGroups || group_heads < 0) return ATTN_ERR_DIMS;
  std::lock_guard<std::mutex> lk(g_order_mu);
  g_force_order = order;
  g_force_group_heads = group_heads;
  return ATTN_OK;
}

extern "C" int attn_diag_fwd_schedule(int BH, int Nq, int Nk, int causal, int q_offset, int k_offset,
                                      long long kv_key_bytes, int launch_kind, int num_sms, int* info, int* seq,
                                      long long seq_len) {
  if (!info) return ATTN_ERR_NULL;
  if (BH < 1 || Nq < 1 || Nk < 1 || num_sms < 1 || kv_key_bytes < 1 || launch_kind < 0 || launch_kind > 2)
    return ATTN_ERR_DIMS;
  const long long qblocks = (static_cast<long long>(Nq) + kBlockM - 1) / kBlockM;
  if (Nq >= kMaxSeq || Nk >= kMaxSeq || static_cast<long long>(BH) * qblocks > INT_MAX) return ATTN_ERR_OVERFLOW;
  FwdParams p;
  fill_params(p, BH, Nq, Nk, causal, q_offset, k_offset, 1, 1.f, num_sms, kv_key_bytes, launch_kind == 1,
              launch_kind == 2);
  const int G = grid_for(p, num_sms);
  int rounds = 0;
  for (int c = 0; c < G; ++c) {
    int round = 0;
    while (unit_for_round(round, p, G, c) != kNoMoreUnits) ++round;
    if (round > rounds) rounds = round;
  }
  info[0] = p.order;
  info[1] = p.group_heads;
  info[2] = G;
  info[3] = rounds;
  info[4] = static_cast<int>(std::llround(predicted_makespan(p, num_sms)));
  info[5] = p.sched_table;
  info[6] = p.pair_tail;
  if (seq) {
    if (seq_len < static_cast<long long>(G) * rounds) return ATTN_ERR_WORKSPACE;
    for (int c = 0; c < G; ++c) {
      bool done = false;
      for (int r = 0; r < rounds; ++r) {
        const int u = done ? kNoMoreUnits : unit_for_round(r, p, G, c);
        done = done || u == kNoMoreUnits;
        // the second half of a pair-tail unit (the sending CTA) as -3 - u
        seq[static_cast<long long>(c) * rounds + r] = (u >= 0 && tail_role(r, p, G, c) == 2) ? -3 - u : u;
      }
    }
  }
  return ATTN_OK;
}

extern "C" int attn_selftest_wait_timeout(void* stream) {
  int dev = 0;
  int rc = device_setup(&dev);
  if (rc != ATTN_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  wait_selftest_kernel<<<1, 32, 0, s>>>(g_timeout_ns, g_dev[dev].err_ptr);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  return attn_check_device_errors(stream, nullptr);
}

// ---------------------------------------------------------------------------
// Split-K/V attention for callers that cannot allocate device memory.
//
// Some callers may not request device memory at all: a serving loop whose
// memory is owned by another allocator (a framework's caching allocator or a
// pool reserved at start-up) and which has no handle on it, or a latency-critical
// path where a cudaMalloc, which can synchronise the device, is not acceptable.
// For them this entry point takes its scratch from a fixed array compiled into
// the library instead of from the caller.
//
// The array is a file-scope __device__ variable of kStaticScratchBytes: every GPU
// that loads the library holds it until the process exits.  Host code cannot use
// the variable's name as a device address; its address is obtained once per
// device with cudaGetSymbolAddress (with that device current) the first time the
// entry point runs there, so the first call on each device should happen before
// any stream capture.  All calls share the one array and it keeps the contents
// of the last call: the kernels overwrite every partial result they later read,
// so nothing has to be cleared, but two calls that overlap on the GPU (e.g. on
// different streams) race on it and must not be issued.
// ---------------------------------------------------------------------------
namespace {
constexpr size_t kStaticScratchBytes = static_cast<size_t>(32) << 20;  // 32 MiB
__device__ __align__(256) unsigned char g_splitkv_static_scratch[kStaticScratchBytes];

struct StaticScratch {
  std::once_flag once;
  int status = ATTN_ERR_CUDA;
  void* ptr = nullptr;
};
StaticScratch g_static_scratch[kMaxDevices];
}  // namespace

extern "C" int attn_fwd_splitkv_static(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                       int H, int Nq, int Nk, int d, int causal, float scale, int num_splits,
                                       void* stream) {
  int rc = validate_tensors(q, k, v, o, lse, B, H, Nq, Nk, d, scale);
  if (rc != ATTN_OK) return rc;
  if (num_splits < 1 || num_splits > kMaxMergeParts) return ATTN_ERR_DIMS;
  int dev = 0;
  if ((rc = device_setup(&dev)) != ATTN_OK) return rc;
  StaticScratch& sc = g_static_scratch[dev];
  std::call_once(sc.once, [&sc] {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_splitkv_static_scratch) == cudaSuccess && ptr != nullptr) {
      sc.ptr = ptr;
      sc.status = ATTN_OK;
    }
  });
  if (sc.status != ATTN_OK) return sc.status;
  // the number of splits attn_fwd_splitkv will use (the same rule), and the
  // scratch those need
  const int s_eff = split_plan((Nk + kBlockN - 1) / kBlockN, num_splits).num_splits;
  if (splitkv_workspace_bytes(static_cast<long long>(B) * H, Nq, d, s_eff) > kStaticScratchBytes)
    return ATTN_ERR_SCRATCH;
  return attn_fwd_splitkv(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale, num_splits, sc.ptr,
                          kStaticScratchBytes, stream);
}

extern "C" size_t attn_splitkv_static_scratch_bytes(void) { return kStaticScratchBytes; }
