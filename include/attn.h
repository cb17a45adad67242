/*
 * attn.h -- C ABI of libattn.so: exact attention forward pass on one NVIDIA
 * GB300 (sm_103a).
 *
 * Operation (the standard scaled dot-product attention that FlashAttention-2
 * reproduces exactly: FlashAttention-2 article, introduction and "Background";
 * computed tile by tile with the online softmax of the ring-attention page,
 * "technical insight", and the deferred rescaling of the news article
 * "FlashAttention scaling, multi-GPU training and weight quantisation", section 1):
 *
 *   for every batch b, head h and query row i:
 *     s_ij   = scale * sum_c q[b,h,i,c] * k[b,h,j,c]      (j = 0 .. N-1)
 *     causal: s_ij = -inf for j > i   (square mask, top-left aligned)
 *     o[b,h,i,:] = sum_j softmax_j(s_i.) * v[b,h,j,:]
 *     lse[b,h,i] = ln sum_j exp(s_ij)                     (natural log)
 *
 * Layouts: q, k, v, o are contiguous [B, H, N, d] (row-major, d fastest);
 * lse is contiguous [B, H, N] float32.
 *
 * Ownership and synchronisation: the caller owns every buffer (device memory)
 * and the stream.  Calls are asynchronous on `stream` (a cudaStream_t; NULL is
 * the legacy default stream); o and lse are valid once the stream has reached
 * the end of the call.  The library allocates no device memory per call and
 * keeps only per-device cached properties and kernel attributes.
 *
 * Errors: arguments are validated before anything is launched; a failed check
 * returns a negative attn_status and launches nothing.  A failure to launch
 * returns ATTN_ERR_LAUNCH.  Inside the kernels every wait on another warp or on
 * a copy engine is bounded (attn_set_wait_timeout_ns); a wait that runs out
 * records ATTN_ERR_TIMEOUT in a device error word, which
 * attn_check_device_errors() reports.  There is no CPU fallback: without an
 * sm_103 device the calls return ATTN_ERR_ARCH or ATTN_ERR_CUDA.
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_NULL = -1,                /* a required pointer is NULL */
  ATTN_ERR_DIMS = -2,                /* a size or count out of range (B, H or N < 1, ...) */
  ATTN_ERR_UNSUPPORTED_HEADDIM = -3, /* d not in {64, 128} */
  ATTN_ERR_DTYPE = -4,               /* dtype not an attn_dtype value */
  ATTN_ERR_ALIGN = -5,               /* q/k/v/o not 16-byte aligned, or lse/scales not 4-byte aligned */
  ATTN_ERR_OVERFLOW = -6,            /* sizes exceed the 32-bit work indexing or TMA limits */
  ATTN_ERR_LAUNCH = -7,              /* the kernel launch failed */
  ATTN_ERR_TIMEOUT = -8,             /* a bounded in-kernel wait ran out (see attn_check_device_errors) */
  ATTN_ERR_ARCH = -9,                /* the current device is not sm_103 */
  ATTN_ERR_SCALE = -10,              /* scale not finite and > 0 */
  ATTN_ERR_CUDA = -11,               /* a CUDA runtime/driver call failed (e.g. no device) */
  ATTN_ERR_SCRATCH = -12,            /* attn_fwd_splitkv_static: the problem needs more than its fixed scratch */
  ATTN_ERR_WORKSPACE = -13           /* a caller-supplied workspace is smaller than its *_workspace_bytes() */
} attn_status;
/*
 * Codes 0 .. -9 are the boundary's base set.  The four later codes refine cases
 * that the base set files under one of its own codes; a caller that only knows
 * the base set can map them back:
 *   ATTN_ERR_SCALE     (-10) -> ATTN_ERR_DIMS   an invalid scalar argument
 *   ATTN_ERR_CUDA      (-11) -> ATTN_ERR_ARCH   no usable sm_103 device (a CUDA
 *                                              call failed before any launch)
 *   ATTN_ERR_SCRATCH   (-12) -> ATTN_ERR_OVERFLOW  the problem exceeds a fixed
 *                                              size limit of the library
 *   ATTN_ERR_WORKSPACE (-13) -> ATTN_ERR_DIMS   a buffer size argument too small
 *
 * `stream` is declared void* so that this header needs no CUDA include: pass a
 * cudaStream_t (the same pointer); NULL is the legacy default stream.
 */

typedef enum { ATTN_BF16 = 0 } attn_dtype;

/*
 * attn_fwd -- BF16 exact attention forward.
 *   q, k, v : const bf16 [B,H,N,d], 16-byte aligned device pointers
 *   o       : bf16 [B,H,N,d] output, 16-byte aligned
 *   lse     : float32 [B,H,N] output, 4-byte aligned; may be NULL (not written)
 *   B, H, N : >= 1;  d : 64 or 128
 *   causal  : 0 = no mask, nonzero = key j visible to query i iff j <= i
 *   scale   : finite, > 0 (usually 1/sqrt(d))
 *   dtype   : ATTN_BF16
 *   stream  : cudaStream_t
 * Arithmetic: bf16 Q K^T and P V on the tensor cores with fp32 accumulation,
 * softmax in fp32 with P rounded to bf16, O rounded to bf16 (nearest-even).
 * Deterministic: the same inputs and shape give the same bits on every call.  A
 * non-causal launch whose last round of work units holds at most one unit per
 * pair of CTAs splits those units' keys over two CTAs (a cluster) and merges the
 * halves (attn_diag_fwd_schedule shows it; attn_diag_set_pair_tail(0) turns it off).
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
             int causal, float scale, int dtype, void* stream);

/*
 * attn_fwd_fp8 -- block-scaled FP8 exact attention forward (FlashAttention-3's
 * FP8 path with block quantisation, news article section 1).
 *   q8, k8, v8 : const e4m3 codes (OCP FP8 E4M3) [B,H,N,d], 16-byte aligned
 *   q_scale, k_scale, v_scale : const float32 [B,H,ceil(N/128)], 4-byte aligned,
 *                finite and > 0: the value of element [b,h,n,c] is
 *                decode(x8[b,h,n,c]) * x_scale[b,h,n/128]
 *   o          : bf16 [B,H,N,d] output;  lse : float32 [B,H,N] or NULL
 *   d          : 128 (other head dimensions return ATTN_ERR_UNSUPPORTED_HEADDIM)
 *   other arguments as attn_fwd.
 * Arithmetic: e4m3 Q K^T on the FP8 tensor cores (fp32 accumulation), softmax in
 * fp32 on the dequantised scores; P rounded to f16 and V's e4m3 codes widened
 * exactly to f16 on chip, P V on the 16-bit tensor path (an e4m3 P loses too much
 * once V has outlier channels); O rounded to bf16.  Deterministic, and non-causal
 * launches may split their last round over CTA pairs, as attn_fwd.
 */
int attn_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* q_scale, const float* k_scale,
                 const float* v_scale, void* o, float* lse, int B, int H, int N, int d, int causal, float scale,
                 void* stream);

/*
 * attn_fwd_partial -- BF16 attention of queries against ONE key/value shard,
 * returning the shard's partial result for an exact merge (the blockwise
 * accumulation of the ring-attention page, "technical insight").
 *   q          : bf16 [B,H,Nq,d]   (query i sits at position q_offset + i)
 *   k, v       : bf16 [B,H,Nk,d]   (key j sits at position k_offset + j)
 *   causal     : nonzero = key j visible to query i iff k_offset + j <= q_offset + i
 *   o_part     : float32 [B,H,Nq,d] output: O over this shard, normalised by the
 *                shard's own softmax sum (16-byte aligned)
 *   lse_part   : float32 [B,H,Nq] output: ln of the shard's sum of exp(scores);
 *                a row with no visible key gets o_part = 0 and lse_part = -inf
 *   q_offset, k_offset : >= 0;  d : 64 or 128;  other arguments as attn_fwd.
 */
int attn_fwd_partial(const void* q, const void* k, const void* v, float* o_part, float* lse_part, int B, int H,
                     int Nq, int Nk, int d, int causal, int q_offset, int k_offset, float scale, void* stream);

/*
 * attn_merge -- exact merge of num_parts partial results over disjoint key sets:
 *   lse = ln sum_s exp(lse_s),  O = sum_s exp(lse_s - lse) O_s.
 *   o_parts, lse_parts : HOST arrays of num_parts (1..16) DEVICE pointers to
 *                        float32 [B,H,N,d] (16-byte aligned) and [B,H,N]
 *   o        : output [B,H,N,d], bf16 (out_fp32 = 0) or float32 (out_fp32 != 0);
 *              may be o_parts[0] when out_fp32 (in-place running merge)
 *   lse      : float32 [B,H,N] output or NULL; may be lse_parts[0]
 * Rows whose partials are all empty (lse = -inf) get O = 0 and lse = -inf.
 */
int attn_merge(const float* const* o_parts, const float* const* lse_parts, int num_parts, void* o, float* lse,
               int out_fp32, int B, int H, int N, int d, void* stream);

/*
 * attn_fwd_splitkv -- BF16 attention with the keys split into num_splits
 * contiguous ranges processed as separate work units (more parallelism when
 * there are few query tiles), followed by attn_merge.
 *   q : bf16 [B,H,Nq,d];  k, v : bf16 [B,H,Nk,d];  o : bf16 [B,H,Nq,d];
 *   lse : float32 [B,H,Nq] or NULL
 *   causal : the queries are the LAST Nq positions of the Nk keys (query i at
 *            position Nk - Nq + i; requires Nq <= Nk); Nq = Nk is attn_fwd's mask
 *   num_splits : 1..16 (reduced if there are fewer 128-key blocks)
 *   workspace : device scratch of at least attn_splitkv_workspace_bytes(...)
 *               bytes (else ATTN_ERR_WORKSPACE), 16-byte aligned, owned by the
 *               caller; its contents on entry do not matter
 */
int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                     int Nk, int d, int causal, float scale, int num_splits, void* workspace,
                     size_t workspace_bytes, void* stream);

/* Scratch bytes attn_fwd_splitkv needs (0 for invalid arguments). */
size_t attn_splitkv_workspace_bytes(int B, int H, int Nq, int d, int num_splits);

/*
 * attn_fwd_splitkv_static -- attn_fwd_splitkv without a workspace argument, for
 * callers that cannot allocate device memory.  The pages have no counterpart:
 * this is a convenience of the library, not part of the method.
 *
 * Who needs it: code that may not request device memory itself -- for example a
 * serving loop whose GPU memory belongs to another allocator (a framework's
 * caching allocator, or a pool reserved at start-up) and which holds no handle
 * on it, or a latency-critical path where cudaMalloc, which can synchronise the
 * device, is not allowed.  Such a caller passes only inputs and outputs; the
 * scratch for the partial results comes from a fixed array compiled into the
 * library (attn_splitkv_static_scratch_bytes() bytes, 32 MiB), which every GPU that
 * loads the library holds until the process exits.
 *
 * Arguments as attn_fwd_splitkv.  Returns ATTN_ERR_SCRATCH, launching nothing,
 * when num_splits * B*H*Nq * (d + 1) * 4 bytes exceed that size (num_splits as
 * reduced to the number of 128-key blocks).  Nothing in this function allocates
 * memory.  The first call on a device looks up the array's device address; make
 * that first call before any stream capture.  Under CUDA's default lazy module
 * loading the library's device code, this array included, is loaded onto a
 * device by the first library call that needs it there (for any entry point),
 * which reserves the 32 MiB and may synchronise: make one library call on each
 * device at start-up, not on a latency-critical path.  All calls share the array (it keeps
 * the last call's contents; every value is rewritten before it is read, so nothing
 * needs clearing): calls whose kernels may overlap on the GPU, such as calls on
 * two streams without ordering between them, race on it and must be avoided.
 */
int attn_fwd_splitkv_static(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                            int Nq, int Nk, int d, int causal, float scale, int num_splits, void* stream);

/* Size in bytes of the fixed scratch attn_fwd_splitkv_static uses. */
size_t attn_splitkv_static_scratch_bytes(void);

/*
 * attn_fwd_host -- attn_fwd with Q, K, V, O and LSE in HOST memory (page-locked
 * for full speed).  The B*H heads go through the device in up to eight chunks of
 * whole heads; the host->device copies of one chunk, the kernel of another and
 * the device->host copies of a third run on separate streams, so the transfers
 * overlap the computation.  Outputs equal those of attn_fwd up to rounding:
 * each chunk is its own launch, and a non-causal launch whose last round is split
 * over CTA pairs (attn_diag_fwd_schedule) merges two key halves of those rows, a
 * different summation order; with the split off (attn_diag_set_pair_tail(0))
 * they are bit for bit those of attn_fwd.
 *   workspace : device scratch of at least attn_fwd_host_workspace_bytes(B,H,N,d)
 *               bytes (else ATTN_ERR_WORKSPACE), 256-byte aligned, owned by the
 *               caller; the call overwrites it
 *   stream    : the kernels run on it; work queued on it after this call sees
 *               the outputs in host memory.  Calls that share a workspace must
 *               be queued on the same stream.
 * Other arguments and errors as attn_fwd (BF16 only).
 */
int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                  int causal, float scale, void* workspace, size_t workspace_bytes, void* stream);

/* Device scratch attn_fwd_host needs (0 for invalid arguments). */
size_t attn_fwd_host_workspace_bytes(int B, int H, int N, int d);

/*
 * attn_fwd_fp8_host -- attn_fwd_fp8 with its inputs and outputs in HOST memory
 * (page-locked for full speed): e4m3 Q, K, V [B,H,N,d] and their fp32 block scales
 * [B,H,ceil(N/128)] in, O bf16 [B,H,N,d] and LSE fp32 [B,H,N] (may be NULL) out.
 * The heads go through the device in up to eight chunks with the copies of one
 * chunk and the kernel of another on separate streams, as attn_fwd_host; each
 * chunk runs attn_fwd_fp8's kernel on whole heads, so the outputs equal those of
 * attn_fwd_fp8 up to rounding (a launch whose last round is split over CTA pairs
 * merges two key halves, as in attn_fwd_host), bit for bit with the split off
 * (attn_diag_set_pair_tail(0)).
 *   workspace : device scratch of at least attn_fwd_fp8_host_workspace_bytes(B,H,N,d)
 *               bytes (else ATTN_ERR_WORKSPACE), 256-byte aligned, owned by the
 *               caller; the call overwrites it
 *   stream    : as attn_fwd_host
 * Returns the codes of attn_fwd_fp8 and attn_fwd_host.
 */
int attn_fwd_fp8_host(const void* q8, const void* k8, const void* v8, const float* q_scale, const float* k_scale,
                      const float* v_scale, void* o, float* lse, int B, int H, int N, int d, int causal, float scale,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Device scratch attn_fwd_fp8_host needs (0 for invalid arguments). */
size_t attn_fwd_fp8_host_workspace_bytes(int B, int H, int N, int d);

/*
 * attn_fwd_fp4p_host -- attn_fwd_fp4p with its inputs and outputs in HOST memory
 * (page-locked for full speed), in the layouts of attn_fwd_fp4p, pipelined in
 * chunks of whole heads as attn_fwd_host; the outputs are bit for bit those of
 * attn_fwd_fp4p.  workspace: at least attn_fwd_fp4p_host_workspace_bytes(B,H,N,d)
 * bytes (else ATTN_ERR_WORKSPACE), 256-byte aligned, owned by the caller.
 * Returns the codes of attn_fwd_fp4p and attn_fwd_host.
 */
int attn_fwd_fp4p_host(const void* q8, const void* k8, const void* vt4, const float* q_scale, const float* k_scale,
                       const uint8_t* vt_scale, void* o, float* lse, int B, int H, int N, int d, int causal,
                       float scale, void* workspace, size_t workspace_bytes, void* stream);

/* Device scratch attn_fwd_fp4p_host needs (0 for invalid arguments). */
size_t attn_fwd_fp4p_host_workspace_bytes(int B, int H, int N, int d);

/*
 * attn_bwd_host -- attn_bwd with Q, K, V, O, dO, LSE, dQ, dK and dV in HOST memory
 * (page-locked for full speed), pipelined in chunks of whole heads as
 * attn_fwd_host (the scratch attn_bwd needs lives in the workspace slots); every
 * chunk runs attn_bwd on whole heads, so the gradients are bit for bit those of
 * attn_bwd.  workspace: at least attn_bwd_host_workspace_bytes(B,H,N,d) bytes
 * (else ATTN_ERR_WORKSPACE), 256-byte aligned, owned by the caller.  Returns the
 * codes of attn_bwd and attn_fwd_host.
 */
int attn_bwd_host(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                  void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale, void* workspace,
                  size_t workspace_bytes, void* stream);

/* Device scratch attn_bwd_host needs (0 for invalid arguments). */
size_t attn_bwd_host_workspace_bytes(int B, int H, int N, int d);

/*
 * attn_fwd_fp4p -- Direct-P FP4 forward (the "Hardware-Aware FP4
 * FlashAttention-4" summary: Direct-P for non-causal inference on Blackwell's
 * FP4 tensor cores).  Q K^T as in attn_fwd_fp8; P V on the FP4 tensor cores with
 * V in MXFP4 and P mapped from the scores straight to e2m1 codes: for every row
 * and every block of 32 keys, E = ceil(max of the block's base-2 scores
 * t = scale log2(e) s_q s_k q.k), code = e2m1 round-to-nearest-even of
 * 2^(t - E + 2), p = value(code) 2^(E - 2); O = sum p v / sum p and
 * lse = ln(sum p).  An approximation of attention (4-bit probabilities).
 *   q8, k8     : e4m3 [B,H,N,d]; q_scale, k_scale fp32 [B,H,N/128] as attn_fwd_fp8
 *   vt4        : V^T as MXFP4 codes, uint8 [B,H,d,N/2] (key 2i in the low nibble
 *                of byte i), 16-byte aligned
 *   vt_scale   : E8M0 block scales of vt4, uint8 [B,H,d,N/32] (value 2^(byte-127)
 *                for keys 32k..32k+31 of channel c), 4-byte aligned
 *   o, lse     : bf16 [B,H,N,d] and fp32 [B,H,N] (lse may be NULL)
 *   d = 128; N a multiple of 128 (else ATTN_ERR_DIMS); causal allowed.
 */
int attn_fwd_fp4p(const void* q8, const void* k8, const void* vt4, const float* q_scale, const float* k_scale,
                  const unsigned char* vt_scale, void* o, float* lse, int B, int H, int N, int d, int causal,
                  float scale, void* stream);

/*
 * attn_bwd -- gradients of the BF16 attention forward (the training use the
 * FlashAttention-2 article reports under "Performance"):
 *   dV = P^T dO,  dS = P o (dP - D) with dP = dO V^T and D_i = do_i . o_i,
 *   dQ = scale dS K,  dK = scale dS^T Q,
 * with P recomputed tile by tile from the forward pass's log-sum-exp.
 *   q, k, v, o, dout : const bf16 [B,H,N,d] (o and lse from attn_fwd with the
 *                      same inputs, causal flag and scale), 16-byte aligned
 *   lse              : const float32 [B,H,N]
 *   dq, dk, dv       : bf16 [B,H,N,d] outputs, 16-byte aligned
 *   workspace        : device scratch of at least attn_bwd_workspace_bytes(B,H,N)
 *                      bytes (else ATTN_ERR_WORKSPACE; 16-byte aligned), owned by
 *                      the caller; the call overwrites it
 *   d : 64 or 128; other arguments as attn_fwd.  Deterministic (no atomics).
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
             void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale, void* workspace,
             size_t workspace_bytes, void* stream);

/* Scratch bytes attn_bwd needs (0 for invalid arguments). */
size_t attn_bwd_workspace_bytes(int B, int H, int N);

/* Human-readable name of an attn_status value (static storage). */
const char* attn_status_string(int status);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns ATTN_OK, ATTN_ERR_TIMEOUT if a kernel gave up on a bounded
 * wait since the last check (*where_out, if not NULL, receives the code of the
 * wait that gave up), or ATTN_ERR_CUDA.
 */
int attn_check_device_errors(void* stream, int* where_out);

/*
 * Sets the limit of every in-kernel wait launched afterwards (nanoseconds,
 * >= 1000; default 4e9).  Returns ATTN_OK or ATTN_ERR_DIMS.
 */
int attn_set_wait_timeout_ns(unsigned long long ns);

/*
 * Self-test of the bounded wait: launches one CTA that waits on an mbarrier
 * nobody arrives at, with the current wait limit.  The kernel gives up, records
 * the timeout and exits; the call synchronises `stream` and returns what
 * attn_check_device_errors returns (ATTN_ERR_TIMEOUT when the wait is working).
 */
int attn_selftest_wait_timeout(void* stream);

/*
 * attn_measure_exp2_rates -- diagnostics (no counterpart on the pages): the
 * throughput of the two exponentials the forward kernel's softmax uses, in
 * exponentials per SM clock cycle per SM, measured on the current device:
 *   *sfu_per_clk_sm      : ex2.approx on the special-function unit
 *   *fma_poly_per_clk_sm : the FMA-pipe polynomial exponential (two per call)
 * Each is one launch of #SM CTAs of 512 threads running eight independent chains
 * x = 2^-x, timed with the SM cycle counter (longest CTA).  Host output pointers;
 * the call synchronises `stream`.  Returns ATTN_OK, ATTN_ERR_NULL, ATTN_ERR_ARCH,
 * ATTN_ERR_LAUNCH or ATTN_ERR_CUDA.
 */
int attn_measure_exp2_rates(float* sfu_per_clk_sm, float* fma_poly_per_clk_sm, void* stream);

/*
 * attn_eval_exp2 -- diagnostics (no counterpart on the pages): evaluates both
 * exponentials on n device floats x: y_poly = the FMA-pipe polynomial (x clamped
 * to >= -127, 2^floor(x) times a degree-3 fit of 2^f with p(0) = 1, relative
 * error <= 8.6e-5 above 2^-126, +0.0 for x <= -127), y_sfu = ex2.approx.ftz.
 * x, y_poly, y_sfu: device float arrays of n >= 1 elements, 4-byte aligned.
 * Asynchronous on `stream`.  Returns ATTN_OK, ATTN_ERR_NULL, ATTN_ERR_DIMS,
 * ATTN_ERR_ALIGN, ATTN_ERR_ARCH, ATTN_ERR_LAUNCH or ATTN_ERR_CUDA.
 */
int attn_eval_exp2(const float* x, float* y_poly, float* y_sfu, long long n, void* stream);

/*
 * attn_diag_tmem_row_max -- diagnostics (no counterpart on the pages): passes one
 * 128 x 128 f32 tile through tensor memory the way the forward kernel reads its
 * scores.  Row t of `in` is stored into TMEM lane t and loaded back with the
 * load-with-maximum the softmax uses for its row max (tcgen05.ld.red .max);
 * vals[t][c] = the loaded values, row_max[t] = the maximum the load returned;
 * block_max[t][b] (may be NULL) = the maxima of columns 32 b .. 32 b + 31 from
 * the four-group form the Direct-P FP4 softmax uses.
 * in, vals: device float arrays of 128 x 128 (row-major); row_max: 128 device
 * floats; block_max: 128 x 4 device floats; all 4-byte aligned.  One CTA of 128
 * threads that allocates 128 TMEM columns.  Asynchronous on `stream`.  Returns
 * ATTN_OK, ATTN_ERR_NULL, ATTN_ERR_ALIGN, ATTN_ERR_ARCH, ATTN_ERR_LAUNCH or
 * ATTN_ERR_CUDA.
 */
int attn_diag_tmem_row_max(const float* in, float* vals, float* row_max, float* block_max, void* stream);

/*
 * attn_diag_fwd_schedule -- diagnostics (no counterpart on the pages; host only,
 * no GPU work): the order in which the forward kernel's persistent CTAs take
 * their work units for a launch of BH heads of Nq query rows over Nk keys
 * (causal: 0/1; q_offset, k_offset: positions of the first query row and key,
 * as in attn_fwd_partial; kv_key_bytes: bytes of one key's K and V rows, 4 d for
 * BF16, 2 d for e4m3) on num_sms SMs, one key range per unit.  launch_kind: 1
 * for a launch of attn_fwd / attn_fwd_host (BF16), whose causal launches may take
 * their units from a table in shared memory and then use any order; 2 for
 * attn_fwd_fp8 / attn_fwd_fp8_host, which compute their units (head-major or
 * zigzag only) and may split their last round over CTA pairs; 0 for the other
 * entry points (computed units, head-major or zigzag, no split).
 * A unit is a pair of 128-row query tiles of one head: id = head * P + r with
 * P = ceil(Nq / 256) pairs per head; under the causal mask r = 0 is the heaviest
 * pair (the last rows), otherwise the first.
 * info (host, 7 ints): [0] order (0 head-major, 1 zigzag, 2 head groups), [1]
 * heads per group, [2] CTAs launched, [3] rounds: the most iterations a CTA
 * takes, [4] the predicted time of the busiest CTA in K/V block periods, [5] 1
 * if the launch takes its units from the table, [6] 1 if the launch splits its
 * last, partly filled round over CTA pairs (clusters of two: the even CTA takes
 * the first half of the unit's key blocks and merges, the odd one the second).
 * seq (host, may be NULL): CTAs x rounds ints, seq[c * rounds + r] = the unit CTA
 * c takes in its r-th iteration (-3 - unit for the odd CTA of a split unit), -2
 * for an iteration it skips, -1 once it is done; seq_len: its capacity in ints
 * (else ATTN_ERR_WORKSPACE).
 * Returns ATTN_OK, ATTN_ERR_NULL, ATTN_ERR_DIMS (also for launch_kind outside
 * 0..2), ATTN_ERR_OVERFLOW or ATTN_ERR_WORKSPACE.
 */
int attn_diag_fwd_schedule(int BH, int Nq, int Nk, int causal, int q_offset, int k_offset, long long kv_key_bytes,
                           int launch_kind, int num_sms, int* info, int* seq, long long seq_len);

/*
 * attn_diag_force_fwd_order -- diagnostics (no counterpart on the pages): makes
 * every later unsplit causal forward launch of this process use the given order
 * (0 head-major, 1 zigzag, 2 head groups of group_heads heads, 0 = all heads in
 * one group) instead of the one the library predicts to balance best; order -1
 * restores the automatic choice.  For tests that run each order on the GPU: a
 * forced order runs from the unit table when the launch qualifies for one (see
 * attn_diag_fwd_schedule), else computed by every role.
 * Returns ATTN_OK or ATTN_ERR_DIMS.
 */
int attn_diag_force_fwd_order(int order, int group_heads);

/*
 * attn_diag_set_pair_tail -- diagnostics (no counterpart on the pages): enable
 * (1, the default) or disable (0) the split of a launch's last, partly filled
 * round over CTA pairs (see attn_diag_fwd_schedule) for every later launch of
 * this process.  For tests and measurements that compare both.  Returns ATTN_OK.
 */
int attn_diag_set_pair_tail(int enable);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */
