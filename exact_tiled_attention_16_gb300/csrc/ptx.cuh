// Thin inline-PTX wrappers for the sm_103a features the attention kernels use:
// mbarriers, TMA tensor loads, tcgen05 tensor-memory allocation, MMA, commit and
// tcgen05.ld/st.  Written from the PTX ISA descriptions of these instructions.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace attn {

// ---------------------------------------------------------------------------
// Error words.  A bounded wait that gives up records where it was and raises
// the CTA-wide abort flag so that the other roles leave their loops quickly.
// ---------------------------------------------------------------------------
enum DeviceError : int {
  kDevErrNone = 0,
  kDevErrTimeout = 1,
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits until the phase with the given parity has completed.  Gives up after
// timeout_ns (or at once when another role has already given up), records the
// failure and returns false.  Never spins unbounded.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t timeout_ns, int* err_word, int where) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > timeout_ns || it > (1u << 30)) {
        *abort_flag = 1;
        if (err_word) atomicCAS(err_word, 0, (where << 8) | kDevErrTimeout);
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Thread-block clusters (CTA pairs): rank, shared::cluster addresses of the
// partner's shared memory, remote stores and mbarrier arrivals with release
// semantics at cluster scope, waits with acquire semantics at cluster scope, and
// the cluster-wide barrier.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The shared::cluster address of `addr` (this CTA's shared memory) in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}
__device__ __forceinline__ void st_cluster_v2(uint32_t addr, float a, float b) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}
__device__ __forceinline__ float4 ld_shared_v4f(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr)
               : "memory");
  return v;
}
// Arrives on an mbarrier in another CTA of the cluster (address from mapa_shared).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t remote_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// mbar_wait for a barrier that another CTA of the cluster arrives on: the same
// bounds, with acquire semantics at cluster scope.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                  uint64_t timeout_ns, int* err_word, int where) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > timeout_ns || it > (1u << 30)) {
        *abort_flag = 1;
        if (err_word) atomicCAS(err_word, 0, (where << 8) | kDevErrTimeout);
        return false;
      }
    }
  }
}
// Every thread of every CTA of the cluster (release before, acquire after).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// TMA: 3-D tiled tensor load global -> shared, completion counted in bytes on
// an mbarrier.  The tensor map lives in kernel parameter space.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0,
                                            int c1, int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}

// TMA: 3-D tiled tensor store shared -> global, tracked by the issuing thread's
// bulk groups.  Box elements outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until every committed bulk group of this thread has read its shared-memory
// source (the buffer may be overwritten), or has completed entirely.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// 16-byte store to shared memory.
// 32 bytes to global memory in one store (sm_100 and later; 32-byte aligned address)
__device__ __forceinline__ void st_global_v8(void* ptr, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(w[0]), "r"(w[1]),
               "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// L2 eviction-priority policies for the TMA cache hint.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------
// Tensor memory (TMEM): 128 lanes x 512 columns of 32-bit cells per SM.
// Address = (lane << 16) | column.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#include "tmem_ldst.inc"

// ---------------------------------------------------------------------------
// tcgen05.mma descriptors.
//
// Shared-memory matrix descriptor (64 bit):
//   [0,14)  start address >> 4
//   [16,30) leading-dimension byte offset >> 4
//   [32,46) stride-dimension byte offset >> 4
//   [46,48) descriptor version = 1
//   [49,52) base offset (0: every operand tile starts 1024-byte aligned)
//   [61,64) layout: 2 = 128-byte swizzle
// For the 128-byte-swizzled layouts used here a "row" is 128 bytes and eight
// rows form a 1024-byte swizzle atom; SBO is the distance between consecutive
// 8-row atoms, LBO the distance between consecutive 128-byte-wide column blocks
// of an MN-major operand.
// ---------------------------------------------------------------------------

// The descriptor split in two 32-bit words: the low word carries the start
// address and LBO (the only fields that change from one MMA step to the next),
// the high word SBO, the version and the layout (constants).
__host__ __device__ constexpr uint32_t sdesc_hi_sw128(uint32_t sbo_bytes) {
  return ((sbo_bytes >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);
}
__device__ __forceinline__ uint32_t sdesc_lo(uint32_t saddr, uint32_t lbo_bytes) {
  return ((saddr >> 4) & 0x3FFFu) | (((lbo_bytes >> 4) & 0x3FFFu) << 16);
}

// A whole 64-bit descriptor (the format above) for a K-major operand in the
// 64-byte swizzled layout (the TMA SWIZZLE_64B image of a tile with 64-byte
// rows): eight rows form a 512-byte atom; layout code 4.
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t saddr, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 4ull << 61;
  return d;
}

// Instruction descriptor (32 bit) of a dense tcgen05.mma:
//   [4,6) D format (1 = f32)   [7,10) A format   [10,13) B format
//   [15] A major (0 = K-major)  [16] B major (1 = MN-major)
//   [17,23) N >> 3              [24,29) M >> 4
// A/B format codes: kind::f16 -> 0 f16, 1 bf16; kind::f8f6f4 -> 0 e4m3, 1 e5m2.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t M, uint32_t N, uint32_t ab_format, bool b_mn_major) {
  return (1u << 4) | (ab_format << 7) | (ab_format << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((N >> 3) << 17) | ((M >> 4) << 24);
}

// tcgen05.mma with shared-memory operands given by descriptor low words and a
// shared constant high word (joined to 64 bits inside the asm):
//   _ss: D[tmem] (+)= A[smem] B[smem]^T;  _ts: D[tmem] (+)= A[tmem] B[smem], A as
//   M x K with row m in lane m and two 16-bit K elements per 32-bit column.
// kind::f16 (bf16 or f16 operands) or kind::f8f6f4 (e4m3), fp32 accumulate.
//
// Every MMA and commit wrapper is called by all 32 lanes of one warp in
// converged, warp-uniform control flow, and one lane chosen by elect.sync issues
// the instruction (always the same lane, so a commit covers every MMA before it).
// Kept warp-uniform, the operands can live in uniform registers: measured, a
// thread issuing alone spends ~48 cycles per MMA, the elected form ~25-30,
// against 64 cycles of tensor-core work for a 128 x 128 x 16 step.
__device__ __forceinline__ void mma_f16_ss_w(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t hi,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b64 da, db;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "mov.b64 da, {%1, %3};\n\tmov.b64 db, {%2, %3};\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_f16_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t hi,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b64 db;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "mov.b64 db, {%2, %3};\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(hi), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_f8_ss_w(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t hi,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b64 da, db;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "mov.b64 da, {%1, %3};\n\tmov.b64 db, {%2, %3};\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Block-scaled FP4 (MXFP4: e2m1 elements, one E8M0 scale per 32 K elements),
// kind::mxf4, scale_vec::2X, K = 64 per instruction, both operands K-major.
// Instruction descriptor: [4,6) B scale-factor id, [7,10) A format (e2m1 = 1),
// [10,13) B format, [17,23) N >> 3, [23] scale format (1 = E8M0), [24,29)
// M >> 4, [29,31) A scale-factor id.  The id selects the byte of the 32-bit
// scale words where this instruction's two scales start: 0 for K elements
// 0..63 of a 128-element row, 2 for 64..127 (1 and 3 are not valid for 2X).
// Scale words in TMEM: for row r of A (and of B), the word holding its four
// 32-element block scales sits in column base + r / 32 of lane r % 32 of the
// lane quadrant the MMA reads, for A the row's own lane, for B every quadrant.
__host__ __device__ constexpr uint32_t make_idesc_mxf4(uint32_t M, uint32_t N, uint32_t sf_id) {
  return (sf_id << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24) |
         (sf_id << 29);
}

// D[tmem] (+)= (A[tmem] * sA) (B[smem] * sB)^T with A = 8 e2m1 per 32-bit column
// (element k of a row in bits 4 (k % 8) of column k / 8).
__device__ __forceinline__ void mma_mxf4_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], [%1], %2, %3, [%4], [%5], p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Arrives once on the mbarrier when every tcgen05.mma issued so far by the
// elected lane has completed (warp-uniform call, like the MMA wrappers).
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// ---------------------------------------------------------------------------
// Arithmetic helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Two-lane fp32 arithmetic (one instruction for both lanes).
__device__ __forceinline__ uint64_t pack_f2(float2 a) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a.x), "f"(a.y));
  return r;
}
__device__ __forceinline__ float2 unpack_f2(uint64_t r) {
  float2 a;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a.x), "=f"(a.y) : "l"(r));
  return a;
}
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(pack_f2(a)), "l"(pack_f2(b)), "l"(pack_f2(c)));
  return unpack_f2(d);
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pack_f2(a)), "l"(pack_f2(b)));
  return unpack_f2(d);
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pack_f2(a)), "l"(pack_f2(b)));
  return unpack_f2(d);
}
__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pack_f2(a)), "l"(pack_f2(b)));
  return unpack_f2(d);
}
// a + b rounded towards -infinity
__device__ __forceinline__ float2 fadd2_rm(float2 a, float2 b) {
  uint64_t d;
  asm("add.rm.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pack_f2(a)), "l"(pack_f2(b)));
  return unpack_f2(d);
}

// 2^x for two floats on the FMA pipe, without the special-function unit (which
// the softmax otherwise saturates with one ex2 per score).
//   x is clamped to >= -127;  x = n + f with n = floor(x), f in [0, 1);
//   2^f ~ p(f) = 1 + c1 f + c2 f^2 + c3 f^3;  2^n enters as n added to the
//   exponent field of p(f).
// n: adding 1.5 * 2^23 with rounding towards -infinity leaves kMagic + floor(x)
// exactly (the sum's unit in the last place is 1), with n in the low mantissa
// bits, so (bits << 23) is n << 23 modulo 2^32.
// p: c1..c3 minimise the largest relative error of p(f) / 2^f on [0, 1] with the
// constant term fixed at 1 (Remez exchange; csrc/fit_exp2_poly.py, which prints
// these float32 values): 8.6e-5 at most in float32 Horner form, below bf16's
// rounding step (2^-9).  p(0) = 1 exactly makes x <= -127 (and x = -inf, a
// masked score) give bits 0x3F800000 - (127 << 23) = 0, i.e. +0.0; for x in
// (-127, -126) the result is a subnormal below 2^-126 (not 2^x, but as
// negligible).  x is at most a few tens here, far from overflow.
constexpr float kExp2PolyC1 = 0x1.63e658p-1f;   // 0.695116758
constexpr float kExp2PolyC2 = 0x1.d2378ap-3f;   // 0.227644995
constexpr float kExp2PolyC3 = 0x1.3baaa6p-4f;   // 0.0770670399
__device__ __forceinline__ float2 exp2_poly2(float2 x) {
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
  x = make_float2(fmaxf(x.x, -127.f), fmaxf(x.y, -127.f));
  const float2 j = fadd2_rm(x, make_float2(kMagic, kMagic));         // kMagic + floor(x)
  const float2 f = fadd2(x, fsub2(make_float2(kMagic, kMagic), j));  // x - floor(x), exact
  float2 p = ffma2(f, make_float2(kExp2PolyC3, kExp2PolyC3), make_float2(kExp2PolyC2, kExp2PolyC2));
  p = ffma2(p, f, make_float2(kExp2PolyC1, kExp2PolyC1));
  p = ffma2(p, f, make_float2(1.f, 1.f));
  return make_float2(__uint_as_float(__float_as_uint(p.x) + (__float_as_uint(j.x) << 23)),
                     __uint_as_float(__float_as_uint(p.y) + (__float_as_uint(j.y) << 23)));
}

// Two floats -> packed bf16x2 (round to nearest even); `lo` lands in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Packed bf16x2 -> two floats (exact); bits 0..15 -> .x
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}
// Two floats -> packed f16x2 (round to nearest even); `lo` lands in bits 0..15.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Two e4m3 codes (byte 0 = first element) -> f16x2 (exact).
__device__ __forceinline__ uint32_t cvt_e4m3x2_to_f16x2(uint16_t codes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(codes));
  return r;
}
// Makes this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA, tcgen05.mma) before it signals a consumer.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Two floats -> two e2m1 codes in one byte (round to nearest even, saturating to
// +-6); `lo` lands in bits 0..3.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Twice the sum of the eight e2m1 values held by a word of non-negative codes
// (nibble k = code of element k), added to acc: a byte-permute table lookup of
// 2 * value (0, 1, 2, 3, 4, 6, 8, 12 for codes 0..7), four bytes at a time, and
// a four-way byte dot product.  Exact integers.
__device__ __forceinline__ uint32_t e2m1x8_sum2(uint32_t word, uint32_t acc) {
  const uint32_t lo = __byte_perm(0x03020100u, 0x0C080604u, word);
  const uint32_t hi = __byte_perm(0x03020100u, 0x0C080604u, word >> 16);
  acc = __dp4a(lo, 0x01010101u, acc);
  return __dp4a(hi, 0x01010101u, acc);
}
// Four code bytes (each in the low byte of a word) -> one word, b0 lowest.
__device__ __forceinline__ uint32_t pack_bytes4(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  return __byte_perm(__byte_perm(b0, b1, 0x0040u), __byte_perm(b2, b3, 0x0040u), 0x5410u);
}
// 2^n for an integer-valued float n (exact; 0 below 2^-126).
__device__ __forceinline__ float exp2_int(float n) {
  return n < -126.f ? 0.f : __int_as_float((static_cast<int>(n) + 127) << 23);
}

}  // namespace attn
