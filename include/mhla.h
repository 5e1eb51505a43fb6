/*
 * mhla.h -- C ABI of libmhla.so: the forward pass of token-level multi-head
 * linear attention (MHLA) on one NVIDIA GB300 (sm_103a).
 *
 * The operation ("MHLA: Restoring Expressivity of Linear Attention via
 * Token-Level Multi-Head", overall framework, flowchart and key design 2):
 *   phi(x) = ELU(x) + 1 applied to Q and K;
 *   the N tokens of a (T, Hg, Wg) grid are split into M non-overlapping
 *   (bt, bh, bw) blocks; for every block b
 *       S_b = sum_{j in b} phi(K_j) V_j^T   (d x d)
 *       z_b = sum_{j in b} phi(K_j)         (d)
 *   the summaries are mixed per query block i with a coefficient matrix Mc:
 *       S~_i = sum_b Mc[i,b] S_b,   z~_i = sum_b Mc[i,b] z_b
 *   and every query q in block i produces
 *       DIVISIVE: o = phi(q)^T S~_i / phi(q)^T z~_i
 *       NONE:     o = phi(q)^T S~_i          (normaliser dropped, key design 2)
 *       MALA:     s = phi(q)^T z~_i, beta = 1 + 1/s, gamma = s / n~_i,
 *                 o = beta phi(q)^T S~_i - gamma v~_i
 *   where v~_i = sum_b Mc[i,b] sum_{j in b} V_j and n~_i = sum_b Mc[i,b] |b|
 *   ("Rectifying Magnitude Neglect in Linear Attention", key designs: the
 *   linear form of MALA, with each global sum replaced by its mixed
 *   counterpart; at M = 1 and Mc = [[1]] it is that page's formula).
 *
 * Conventions shared by every call:
 *   - Q, K, V and out are contiguous [B, H, N, d] arrays, d innermost, tokens
 *     in raster order of the grid: t = (tau * Hg + y) * Wg + x.
 *   - Blocks are numbered in raster order of the block grid
 *     (T/bt, Hg/bh, Wg/bw); Mc is a float32 [M, M] row-major array whose row
 *     is the query block and whose column is the summary block.  One Mc is
 *     shared by all batches and heads.
 *   - dtype BF16: Q, K, V, out hold bf16 values; F32: float32.
 *   - Pointers passed to mhla_forward are device pointers owned by the
 *     caller; the library never frees them and keeps none of them after the
 *     call returns.  Q, K, V and out must be 16-byte aligned, the workspace
 *     256-byte aligned, Mc 4-byte aligned.
 *   - The stream argument is a cudaStream_t (NULL = legacy default stream).
 *     Work is enqueued asynchronously; no call synchronises the host unless
 *     its comment says so.
 *   - Every argument is checked on the host before anything is enqueued.  An
 *     invalid argument returns an error status and enqueues nothing.  No
 *     kernel traps.  A kernel whose bounded wait on the device expires stops
 *     early and records MHLA_ERR_DEVICE_TIMEOUT, which mhla_device_status
 *     reports; the output of that call is then undefined.
 *   - The library keeps per-device state (cached tensor-map encoder, device
 *     error word); calls from several host threads on the same device are
 *     safe except mhla_set_phase_events, which is process-wide.
 */
#ifndef MHLA_H_
#define MHLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MHLA_ABI_VERSION 3

typedef enum mhla_status {
  MHLA_OK = 0,
  MHLA_ERR_INVALID_ARG = 1,     /* bad pointer, shape, enum or alignment      */
  MHLA_ERR_UNSUPPORTED = 2,     /* valid request the library does not support */
  MHLA_ERR_WORKSPACE = 3,       /* workspace missing or smaller than required */
  MHLA_ERR_CUDA = 4,            /* a CUDA runtime call failed                  */
  MHLA_ERR_DEVICE_TIMEOUT = 5,  /* a kernel's bounded wait expired             */
  MHLA_ERR_OVERFLOW = 6         /* reserved: no kernel reports it since ABI 3  */
} mhla_status;

typedef enum mhla_dtype { MHLA_DTYPE_BF16 = 0, MHLA_DTYPE_F32 = 1 } mhla_dtype;

/* ELU1: phi(x) = x + 1 (x > 0), exp(x) (x <= 0).  IDENTITY: phi(x) = x; for
 * tests only, the caller keeps the features positive. */
/* Feature map phi applied to Q and K.  ELU1: ELU(x) + 1 (alpha = 1); RELU:
 * max(x, 0); EXP: e^x, evaluated in float32 without a shift (inputs whose
 * exponential overflows float32 give inf/NaN) -- the three maps of "Rectifying
 * Magnitude Neglect in Linear Attention", ablations.  IDENTITY (phi(x) = x) is
 * for tests that keep features positive.  A query whose denominator
 * s = phi(q)^T z~_i is exactly zero (ReLU features, or a zero row of Mc) gets
 * output 0 under DIVISIVE and MALA, and no gradient. */
typedef enum mhla_feature_map {
  MHLA_FEATURE_ELU1 = 0,
  MHLA_FEATURE_IDENTITY = 1,
  MHLA_FEATURE_RELU = 2,
  MHLA_FEATURE_EXP = 3
} mhla_feature_map;

typedef enum mhla_norm { MHLA_NORM_DIVISIVE = 0, MHLA_NORM_MALA = 1, MHLA_NORM_NONE = 2 } mhla_norm;

/* AUTO picks MULTIPASS for bf16 with d = 64, SIMT otherwise.
 * SIMT:      CUDA-core kernels, float32 arithmetic, any supported d, both dtypes.
 * MULTIPASS: tcgen05/TMEM tensor-core kernels fed by TMA (bf16, d = 64):
 *            block summaries -> mixing GEMM -> output with fused epilogue.
 *            For the DIVISIVE and NONE norms the mixing multiplies fp16
 *            operands: each block summary's S_b and z_b are stored times
 *            their own power of two (the part's largest entry lands in
 *            [2^14, 2^15)), and a small kernel folds those exponents into a
 *            per-head fp16 copy of Mc whose rows are scaled so that each
 *            row's largest entry lies in [0.5, 1); the output step applies
 *            the remaining power of two.  So every finite input stays in
 *            range: a summary entry keeps full fp16 precision down to 2^-29
 *            of its part's largest entry, and a mixed term down to 2^-24 of
 *            its row's largest term.  MALA (and the causal form) mix bf16
 *            high + low parts, which have the float32 range.
 * FUSED:     the MULTIPASS kernels as three groups of CTAs in one
 *            cooperative launch that work through the heads concurrently;
 *            the stack and the mixed summaries live in a ring of a few heads
 *            that stays in L2, so less workspace.  Every norm mixes bf16
 *            high + low parts here (same results as MULTIPASS under MALA;
 *            within the same tolerance otherwise).  Needs a device with
 *            cooperative launch; the split of the SMs between the groups
 *            follows a work estimate, and the environment variable
 *            MHLA_FUSED_GROUPS="s,x,o" (CTA counts) overrides it for
 *            tuning. */
typedef enum mhla_variant {
  MHLA_VARIANT_AUTO = 0,
  MHLA_VARIANT_SIMT = 1,
  MHLA_VARIANT_MULTIPASS = 2,
  MHLA_VARIANT_FUSED = 3
} mhla_variant;

/* Memory layout of q, k, v, out (and dout, dq, dk, dv): BHND = [B, H, N, d]
 * (each head's tokens contiguous); BNHD = [B, N, H, d] (token-major, as a
 * fused QKV projection writes it: the H heads of a token are adjacent). */
typedef enum mhla_layout { MHLA_LAYOUT_BHND = 0, MHLA_LAYOUT_BNHD = 1 } mhla_layout;

typedef struct mhla_params {
  int batch;        /* B >= 0                                              */
  int heads;        /* H >= 0                                              */
  int head_dim;     /* d in {16, 32, 64, 128}                              */
  int grid[3];      /* (T, Hg, Wg) token grid, each >= 1; 1D = (1, 1, N)   */
  int block[3];     /* (bt, bh, bw), each >= 1 and dividing grid[i]        */
  int dtype;        /* mhla_dtype                                          */
  int feature_map;  /* mhla_feature_map                                    */
  int norm;         /* mhla_norm                                           */
  int variant;      /* mhla_variant                                        */
  int causal;       /* 0: every token sees every block (the method as the
                     * MHLA page defines it); 1: block-ordered causal form --
                     * tokens ordered by (block, position inside the block),
                     * query t sees keys up to itself: earlier blocks through
                     * the strict lower triangle of Mc, its own block through
                     * Mc[i, i] and only the tokens up to t.  mhla_backward
                     * runs it on the float32 CUDA-core kernels.  AUTO
                     * takes the tensor cores for bf16, d = 64, DIVISIVE or
                     * NONE when every token chunk is a contiguous run of its
                     * block's local order, else the float32 kernels;
                     * MULTIPASS outside that set and FUSED return
                     * MHLA_ERR_UNSUPPORTED.                                 */
  int layout;       /* mhla_layout of the token tensors                    */
  int mc_per_head;  /* 0: mc is [M, M], shared by every (batch, head);
                     * 1: mc is [H, M, M], head h mixes with mc[h] (shared over
                     * the batch) -- mhla_backward's dmc then has the same
                     * shape, summed over the batch only.  Not with
                     * MHLA_VARIANT_FUSED (MHLA_ERR_UNSUPPORTED).           */
} mhla_params;

/* What a call with these parameters will run (for tests and benchmarks). */
typedef struct mhla_plan_info {
  int n_tokens;          /* N                                              */
  int n_blocks;          /* M                                              */
  int block_tokens;      /* n_b = bt * bh * bw                             */
  int variant;           /* the variant AUTO resolved to                   */
  int kernels_per_call;  /* kernel launches one mhla_forward enqueues     */
  int summary_splits;    /* partial summaries per block (long blocks)      */
  size_t workspace_bytes;
} mhla_plan_info;

/* Validates p and fills *info.  Returns MHLA_ERR_INVALID_ARG or
 * MHLA_ERR_UNSUPPORTED for parameters mhla_forward would reject. */
mhla_status mhla_plan(const mhla_params* p, mhla_plan_info* info);

/* Device workspace mhla_forward needs for p, in bytes (0 for an empty
 * problem).  Returns the same errors as mhla_plan. */
mhla_status mhla_workspace_bytes(const mhla_params* p, size_t* bytes);

/* The MHLA forward pass (see the top of this file).
 *   q, k, v     device [B, H, N, d] inputs (dtype p->dtype)
 *   mc          device float32 [M, M] mixing coefficients
 *   out         device [B, H, N, d] output (dtype p->dtype); must not alias
 *               q, k, v, mc or the workspace
 *   workspace   device scratch of at least mhla_workspace_bytes(p) bytes, or
 *               NULL with workspace_bytes == 0, in which case the library
 *               takes stream-ordered memory (cudaMallocAsync) on `stream` and
 *               returns it (cudaFreeAsync) on the same stream
 *   stream      cudaStream_t the kernels are enqueued on
 * B * H * N == 0 is a no-op that returns MHLA_OK.  Non-positive Mc rows or
 * features make the divisive and MALA denominators reach zero; IEEE inf/NaN
 * then propagate (the pages put no epsilon in them). */
mhla_status mhla_forward(const void* q, const void* k, const void* v, const float* mc,
                         const mhla_params* p, void* out, void* workspace,
                         size_t workspace_bytes, void* stream);

/* Allocation-free variant of mhla_forward for callers that cannot allocate
 * device memory when they call (allocator callbacks and out-of-memory
 * handlers, plugin hosts that forbid cudaMalloc after start-up, real-time
 * loops that must not touch the allocator).  The pages have no counterpart:
 * it is the same forward pass, with its scratch memory taken from a 32 MiB
 * static device array inside this library instead of a caller workspace.
 *   q, k, v, mc, p, out, stream   as for mhla_forward
 * Allocates nothing: no cudaMalloc, cudaMallocAsync or cudaFree.  Problems
 * whose mhla_workspace_bytes(p) exceeds 32 MiB return MHLA_ERR_WORKSPACE and
 * enqueue nothing.  Each call looks up the array's device address with
 * cudaGetSymbolAddress for the current device.  The first call on a device
 * may be the one that loads the library's code there (CUDA loads modules
 * lazily by default), and loading commits the array's 32 MiB of device
 * memory at that moment: make a first, small call at start-up, before any
 * stream capture, if later calls must not depend on free device memory.
 * Every GPU that loads the library holds the array until the process exits.
 * All calls on a device share the one array, so calls whose work overlaps on
 * the GPU (different streams, or different host threads) race and must be
 * serialised by the caller.  Nothing in the array has to start at zero: each
 * call overwrites every byte it reads. */
mhla_status mhla_forward_noalloc(const void* q, const void* k, const void* v, const float* mc,
                                 const mhla_params* p, void* out, void* stream);

/* Device buffer mhla_forward_host needs: room for Q, K, V, Mc, out and the
 * workspace, each 256-byte aligned. */
mhla_status mhla_host_buffer_bytes(const mhla_params* p, size_t* bytes);

/* End-to-end call on HOST arrays: copies q, k, v, mc into dev_buffer, runs
 * the forward pass and copies the result into out, then synchronises
 * `stream` and returns.  Large problems are cut into up to 8 groups of
 * (batch, head) units (at least ~32 MB of each input per group): group g's
 * inputs are copied in on one library-owned stream while group g-1's kernels
 * run on `stream` and group g-2's result is copied back on another, ordered
 * by events; everything starts after the work already queued on `stream`.
 * Host arrays have the layouts of mhla_forward; page-locked host memory makes
 * the copies asynchronous DMA transfers.  dev_buffer is a device allocation
 * of at least mhla_host_buffer_bytes(p) bytes.  Calls on the same device are
 * serialised (the copy streams are per device). */
mhla_status mhla_forward_host(const void* q, const void* k, const void* v, const float* mc,
                              const mhla_params* p, void* out, void* dev_buffer,
                              size_t dev_buffer_bytes, void* stream);

/* Backward pass: the gradients of L = sum(dout * o), o = mhla_forward(q, k, v,
 * mc), with respect to q, k, v and mc -- the chain rule of the forward steps
 * ("MHLA: Restoring Expressivity of Linear Attention via Token-Level
 * Multi-Head": Mc is learned end to end, key design 3; the pages print no
 * gradient).  Every norm and feature map of the forward.  p->variant:
 * MHLA_VARIANT_AUTO takes the tensor cores for bf16 with head_dim 64 (split
 * bf16 high + low operands, float32 accumulation) and float32 CUDA-core
 * kernels otherwise; MHLA_VARIANT_SIMT forces the CUDA-core kernels;
 * MULTIPASS and FUSED ask for the tensor cores (MHLA_ERR_UNSUPPORTED where
 * they do not apply).  The forward summaries are recomputed inside the call.
 * p->causal = 1 differentiates the block-ordered causal form on the CUDA
 * cores (AUTO or SIMT; MULTIPASS and FUSED return MHLA_ERR_UNSUPPORTED):
 * Mc above its diagonal does not enter that output, and its dmc entries
 * are 0.
 *   dout, dq, dk, dv: [B, H, N, d] in p->dtype, like q; dmc: float32 [M, M],
 *   overwritten with the sum over every (batch, head).
 * Device pointers, 16-byte aligned (mc, dmc 4-byte); dq, dk, dv, dmc must
 * not overlap the inputs or each other.  workspace as for mhla_forward, of
 * at least mhla_backward_workspace_bytes(p) bytes (NULL with 0 bytes: the
 * library allocates it on `stream`).  Asynchronous on `stream`.  Returns the
 * validation errors of mhla_forward, MHLA_ERR_WORKSPACE, MHLA_ERR_CUDA. */
mhla_status mhla_backward_workspace_bytes(const mhla_params* p, size_t* bytes);
mhla_status mhla_backward(const void* q, const void* k, const void* v, const float* mc, const void* dout,
                          const mhla_params* p, void* dq, void* dk, void* dv, float* dmc, void* workspace,
                          size_t workspace_bytes, void* stream);

/* Reads and clears the device error word of the current device.  Blocks the
 * host until the device is idle.  *code receives MHLA_OK or the first status
 * a kernel recorded (MHLA_ERR_DEVICE_TIMEOUT); *detail
 * receives a kernel-specific location code (0 if none).  Either pointer may
 * be NULL. */
mhla_status mhla_device_status(int* code, int* detail);

/* Timing hook.  With n == MHLA_NUM_PHASE_EVENTS, each later mhla_forward
 * records events[0] before its first kernel and events[i] after phase i
 * (1: Mc preparation, 2: block summaries, 3: folding the fp16 records'
 * exponents into Mc, 4: mixing, 5: output) on its stream; phases a variant
 * does not have record at the same point as the previous one (the fused
 * launch runs phases 2-5 as one kernel, recorded after phase 5).  Events
 * between the kernels serialise them.  events are cudaEvent_t handles owned
 * by the caller.  n == 0 turns the hook off.  Process-wide; not meant for
 * concurrent callers. */
#define MHLA_NUM_PHASE_EVENTS 6
mhla_status mhla_set_phase_events(void* const* events, int n);

/* The same hook for mhla_backward: events[0] before its first kernel, then
 * after each phase (1: forward summaries and mixing recomputed, 2: output
 * step gradients dq, dS~, dz~, 3: gradient mixing dS, dz, 4: dMc, 5: dk, dv).
 * Independent of mhla_set_phase_events; same ownership and rules. */
#define MHLA_NUM_BWD_PHASE_EVENTS 6
mhla_status mhla_set_backward_phase_events(void* const* events, int n);

/* Testing hooks for the FUSED variant's waits on other CTA groups (the pages
 * have no counterpart; a wait that cannot end must be testable without
 * hanging the GPU).
 *   MHLA_DEBUG_FLOW_WAIT_NS  limit of each such wait, in nanoseconds
 *                            (value <= 0 restores the default, one second).
 *   MHLA_DEBUG_FLOW_STALL    value != 0: the output group waits for one more
 *                            mixing signal per head than will ever arrive, so
 *                            its wait expires; every CTA then stops early and
 *                            mhla_device_status reports MHLA_ERR_DEVICE_TIMEOUT
 *                            (the output is not written).  0 turns it off.
 * Returns MHLA_ERR_INVALID_ARG for an unknown option.  Process-wide, read at
 * each launch; not for production use. */
typedef enum mhla_debug_option { MHLA_DEBUG_FLOW_WAIT_NS = 1, MHLA_DEBUG_FLOW_STALL = 2 } mhla_debug_option;
mhla_status mhla_set_debug(int option, long long value);

/* Static description of a status code; never NULL. */
const char* mhla_status_string(mhla_status s);

/* Text of the last CUDA error this thread saw inside the library ("" if none). */
const char* mhla_last_error_string(void);

/* MHLA_ABI_VERSION of the loaded library. */
int mhla_abi_version(void);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* MHLA_H_ */
