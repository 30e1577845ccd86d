/*
 * lapl_attn.h -- C ABI of the GB300 (sm_103a) Laplacian-kernel Nystrom attention forward.
 *
 * The operation ("LaplacianFormer: Rethinking Linear Attention with Laplacian Kernel",
 * explainer pages): for every batch b and head h independently,
 *   L  = 2-D average pooling of K over the grid_h x grid_w token grid into m = s*s rows
 *        (English page, 2.C.1: landmarks selected via average pooling)
 *   A  = exp(-cdist_L1(Q, L) / lambda)        [N, m]   (English page, 2.A: Laplacian kernel)
 *   B  = exp(-cdist_L1(L, K) / lambda)        [m, N]
 *   W  = exp(-cdist_L1(L, L) / lambda) + eps I  [m, m] (English page, 2.C.2: eps I keeps W PD)
 *   X  = T Newton-Schulz steps X <- X (2I - W X), X0 = W^T / (|W|_1 |W|_inf)
 *        (English page, 2.C.2; German page, 2: multiply-only inverse)
 *   A^ = (A - mean_col) / sqrt(var_col + delta) + bias   (Korean page, 2.2: whitening with a
 *        diagonal estimator; mean/var per landmark column over the N tokens, var divides by N)
 *   O  = A^ (X (B V))                         [N, d]   (Chinese page, 2.2: the N x N matrix
 *        is never formed)
 *
 * Layouts: Q, K, V, O are [B, H, N, d] contiguous (C order), token n = r * grid_w + c.
 * Every buffer is owned by the caller.  The handle holds host state only: the configuration,
 * two CUDA events and one auxiliary stream.  After pooling the forward splits into two
 * chains, the Newton-Schulz solve and the distance + B V kernels; the longer one runs on the
 * launching stream, the other on the auxiliary stream, and they join before M = X (B V).  The
 * library's
 * device globals are a 4-byte error word and the scratch of lapl_attn_forward_noalloc.  No
 * entry point allocates device memory; forward() never synchronises the host.
 *
 * Errors: every entry point returns a lapl_status.  Argument errors are detected on the host
 * before any launch.  CUDA errors from launches map to LAPL_ERR_CUDA (the CUDA error string is
 * available from lapl_attn_last_error()).  Nothing aborts the process.
 *
 * Threading: a handle may be used by one host thread at a time, on one stream at a time.
 */
#ifndef LAPL_ATTN_H
#define LAPL_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LAPL_OK = 0,
  LAPL_ERR_INVALID_ARG = 1,     /* null pointer, bad size or parameter                    */
  LAPL_ERR_UNSUPPORTED = 2,     /* valid but outside what the kernels handle (see create) */
  LAPL_ERR_WORKSPACE = 3,       /* workspace smaller than lapl_attn_workspace_size()       */
  LAPL_ERR_ALIGNMENT = 4,       /* a device pointer is not 16-byte aligned                 */
  LAPL_ERR_CUDA = 5,            /* a CUDA runtime call or launch failed                    */
  LAPL_ERR_DEVICE_TIMEOUT = 6,  /* a bounded device-side wait gave up (device_errors)      */
  LAPL_ERR_NOT_IMPLEMENTED = 7
} lapl_status;

typedef enum { LAPL_F32 = 0, LAPL_BF16 = 1 } lapl_dtype;

/*
 * Similarity kernel k(x, y) = exp(-D(x, y) / lambda) of A, B and W.
 *   LAPL_KERNEL_LAPLACIAN: D = sum_c |x_c - y_c| (the method: English page, 2.A).
 *   LAPL_KERNEL_GAUSSIAN:  D = sum_c (x_c - y_c)^2, the Gaussian kernel of earlier linear
 *     attention that the pages set the Laplacian one against (English page, 1 "Theoretical
 *     Mismatch": similarity decaying with the squared l2 distance); a drop-in that keeps every
 *     other step, eps I included.
 */
typedef enum { LAPL_KERNEL_LAPLACIAN = 0, LAPL_KERNEL_GAUSSIAN = 1 } lapl_kernel;

/*
 * How M ~ W^-1 (B V) is obtained.
 *   LAPL_SOLVER_NEWTON_SCHULZ: X = T Newton-Schulz steps, M = X (B V) (the method).
 *   LAPL_SOLVER_CG: M = T conjugate-gradient iterations on W M = B V, each column from zero,
 *     a column stopping early only where no step is defined (r.r = 0 or p.Wp <= 0); X is
 *     not formed.  The solver the pages compare Newton-Schulz with (German page, 4; English
 *     page, 4 "Solver Robustness").  All of its work runs after the B V kernel, on the
 *     launching stream.
 */
typedef enum { LAPL_SOLVER_NEWTON_SCHULZ = 0, LAPL_SOLVER_CG = 1 } lapl_solver;

typedef struct {
  int batch;          /* B >= 0 (B == 0: forward is a no-op)                                */
  int heads;          /* H >= 1                                                             */
  int grid_h, grid_w; /* token grid, N = grid_h * grid_w                                    */
  int head_dim;       /* d: multiple of 8, 8 <= d <= 128                                    */
  int num_landmarks;  /* m = s*s with 1 <= s <= 8; grid_h % s == 0 and grid_w % s == 0      */
  float lambda;       /* kernel scale, > 0 (the pages' best value is 4)                    */
  float eps;          /* >= 0, added to the diagonal of W                                    */
  float delta;        /* > 0 when whiten != 0: variance floor inside the square root         */
  int ns_steps;       /* T, 0 <= T <= 1000: exactly T Newton-Schulz steps (or at most T CG
                         iterations per column with LAPL_SOLVER_CG)                         */
  int whiten;         /* 1: whiten A (default); 0: A^ = A and bias is ignored                */
  int in_dtype;       /* lapl_dtype of Q, K, V                                               */
  int out_dtype;      /* lapl_dtype of O (LAPL_F32 recommended; LAPL_BF16 rounds at the end) */
  int kernel;         /* lapl_kernel (0, the Laplacian kernel, when the struct is zeroed)     */
  int solver;         /* lapl_solver (0, Newton-Schulz, when the struct is zeroed)            */
} lapl_attn_config;

typedef struct lapl_attn_plan* lapl_attn_handle;

/* Nullable device pointers for intermediate results (all fp32, C order). */
typedef struct {
  float* d_ql;       /* [B,H,N,m] raw distances D(Q_i, L_j) (L1 sum_c |Q_ic - L_jc|, or
                        the squared l2 distance for the Gaussian kernel)                    */
  float* d_ll;       /* [B,H,m,m] raw distances between landmarks       */
  float* d_lk;       /* [B,H,m,N] raw distances D(L_j, K_n)             */
  float* landmarks;  /* [B,H,m,d] L                                      */
  float* w;          /* [B,H,m,m] W = k(L,L) + eps I                     */
  float* x;          /* [B,H,m,m] X after T Newton-Schulz steps (not written with CG) */
  float* a;          /* [B,H,N,m] A = k(Q,L), before whitening           */
  float* mu;         /* [B,H,m]   column means of A                      */
  float* rstd;       /* [B,H,m]   1/sqrt(var + delta) (var divides by N) */
  float* bv;         /* [B,H,m,d] B V                                    */
  float* m;          /* [B,H,m,d] M = X (B V), or the CG solution        */
} lapl_attn_debug;

/* Library version: major * 10000 + minor * 100 + patch. */
int lapl_attn_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* lapl_attn_status_string(lapl_status s);

/* Text of the last CUDA error seen by this handle ("" if none; owned by the handle). */
const char* lapl_attn_last_error(lapl_attn_handle h);

/*
 * Validate cfg and create a plan on the current CUDA device.  *out receives the handle.
 * Returns LAPL_ERR_INVALID_ARG / LAPL_ERR_UNSUPPORTED for bad configurations (nothing is
 * created), LAPL_ERR_CUDA if the event/stream creation fails.
 */
lapl_status lapl_attn_create(const lapl_attn_config* cfg, lapl_attn_handle* out);

/* Bytes of device workspace forward() needs (a multiple of 256, linear in B*H*N). */
lapl_status lapl_attn_workspace_size(lapl_attn_handle h, size_t* bytes);

/*
 * Forward pass, stream-ordered and asynchronous on `stream` (a cudaStream_t; NULL = legacy
 * default stream).  q, k, v: device [B,H,N,d] in in_dtype; bias: device [H,m] fp32 or NULL
 * (zeros); out: device [B,H,N,d] in out_dtype; workspace: device, >= workspace_size bytes,
 * contents need not be initialised and are overwritten.  q, k, v, out and workspace must be
 * 16-byte aligned and must not overlap.  No allocation, no host synchronisation.
 */
lapl_status lapl_attn_forward(lapl_attn_handle h, const void* q, const void* k, const void* v,
                              const float* bias, void* out, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * forward() that also keeps in the workspace what lapl_attn_backward needs beyond the forward's
 * own intermediates: every Newton-Schulz iterate X_0 .. X_T and the reduced B V (about 2-3 us
 * more at the stage-1 shape).  Same arguments, results bit for bit equal to forward().
 * LAPL_ERR_UNSUPPORTED with the CG solver.
 */
lapl_status lapl_attn_forward_train(lapl_attn_handle h, const void* q, const void* k,
                                    const void* v, const float* bias, void* out,
                                    void* workspace, size_t workspace_bytes, void* stream);

/* forward() that also writes the non-NULL fields of *dbg (device buffers, fp32). */
lapl_status lapl_attn_forward_debug(lapl_attn_handle h, const void* q, const void* k,
                                    const void* v, const float* bias, void* out,
                                    void* workspace, size_t workspace_bytes, void* stream,
                                    const lapl_attn_debug* dbg);

/*
 * Bytes of device staging memory forward_host() needs: device copies of Q, K, V, O and the
 * workspace, each 256-byte aligned (for a batch of two or more, one such region per half-batch
 * forward, see forward_host()).
 */
lapl_status lapl_attn_host_staging_size(lapl_attn_handle h, size_t* bytes);

/*
 * End-to-end forward from host memory: copies q, k, v (host, in_dtype) and bias (host [H,m]
 * fp32 or NULL) into `staging` (device, >= host_staging_size bytes), runs forward(), and copies
 * O back into out (host, out_dtype), all on `stream`.  Page-locked host buffers make the copies
 * asynchronous; with pageable memory the CUDA runtime stages them synchronously.  Returns
 * after enqueueing: synchronise the stream before reading out.
 * With a batch of two or more the call runs two forwards of half the batch each (the first
 * ceil(B/2) batches on `stream`, the others on a stream of the plan, joined back into `stream`
 * before the call's work ends), so that one half's copies overlap the other's kernels and the
 * first half's output is copied back while the second computes.  The results equal those of
 * forward() bit for bit.  The environment variable LAPL_ATTN_HOST_SPLIT=0, read at create,
 * keeps a single forward.
 */
lapl_status lapl_attn_forward_host(lapl_attn_handle h, const void* q, const void* k,
                                   const void* v, const float* bias, void* out, void* staging,
                                   size_t staging_bytes, void* stream);

/*
 * Stage timing, a profiling aid.  After lapl_attn_set_timing(h, 1) every forward records CUDA
 * events (created here, host-owned) on the stream that runs each kernel (the solve runs on the
 * launching stream and the distance and B V kernels on the side stream when plan_info's
 * ns_exclusive is 1; the other way round otherwise).
 * lapl_attn_stage_times() waits for the events of the last forward (it synchronises the host
 * with them) and writes the elapsed milliseconds of
 *   ms[0] pooling, ms[1] Newton-Schulz, ms[2] distance kernel, ms[3] B V partials, ms[4]
 *   finish (the wait for the solve, then the B V reduction and M = X (B V); with the CG
 *   solver, the CG kernel, W included, and ms[1] is 0), ms[5] output (column statistics,
 *   whitening and O = A^ M).
 * LAPL_ERR_INVALID_ARG if timing is off or no forward ran since it was switched on.
 */
lapl_status lapl_attn_set_timing(lapl_attn_handle h, int enable);
lapl_status lapl_attn_stage_times(lapl_attn_handle h, float* ms);

/*
 * Timeline of the last timed forward (same events as lapl_attn_stage_times, same waiting and
 * errors): milliseconds since the start of the forward on the launching stream of
 *   ms[0] start (0), ms[1] pooling done, ms[2] Newton-Schulz start, ms[3] Newton-Schulz done,
 *   ms[4] distance kernel start (its stream has seen pooling done), ms[5] distance kernel
 *   done, ms[6] B V partials done, ms[7] M = X (B V) done, ms[8] output done.
 */
lapl_status lapl_attn_stage_marks(lapl_attn_handle h, float* ms);

/* Number of kernels one forward launches (for launch accounting): 6, or 5 with the CG
 * solver; one more when B V runs on the tensor cores with whitening on (plan_info
 * bv_tensor_core: the column statistics are then a launch of their own). */
int lapl_attn_kernels_per_forward(lapl_attn_handle h);

/*
 * Device-side failure report.  Kernels that wait on shared-memory barriers (the distance
 * kernel's TMA pipeline, the tensor-core Newton-Schulz solve) bound every such wait (one second
 * by default); a wait that gives up sets a bit of a device error word (one per device, shared
 * by all handles) -- bit 1 the distance kernel, bit 2 the tensor-core solve, bit 4 a tensor-core
 * kernel of the output chain -- and the waiting
 * warps leave the kernel after the copies and tensor-core operations they issued have
 * completed, so a failed forward ends instead of hanging, the context stays usable, and its
 * outputs are undefined.  This call copies the word to *flags, clears it, and synchronises
 * `stream` (a cudaStream_t; enqueue it after the forwards to be checked).  Returns
 * LAPL_ERR_DEVICE_TIMEOUT (with a message naming the kernel in lapl_attn_last_error) when a
 * flag was set, LAPL_OK when none was, LAPL_ERR_CUDA if the copy fails.
 */
lapl_status lapl_attn_device_errors(lapl_attn_handle h, void* stream, unsigned* flags);

/*
 * Fault injection, for testing the failure report above without faulting the GPU (the pages
 * have no counterpart).  wait_ns: the bound of every barrier wait of this plan's distance
 * kernel and tensor-core B V and output kernels (0 restores the default of one second).
 * skip_last_copy names the kernel that never issues the copy of each CTA's last chunk or tile,
 * so that the waits on it run out after wait_ns with nothing else outstanding:
 *   1  the distance kernel: the split-pipe kernel (plan_info cdist_tma = 2; its producer skips
 *      the copy) or the Gaussian tensor-core kernel (cdist_tma = 3; its converter warps never
 *      publish the chunk); reported as bit 1;
 *   2  the tensor-core output kernel (out_tensor_core = 1; its copying thread skips the last
 *      A^T tile); reported as bit 4;
 *   3  the tensor-core B V kernel (bv_tensor_core = 1; its copy warp skips the last tile);
 *      reported as bit 4.
 * Applies to forwards launched after the call.  0 = normal operation; other values return
 * LAPL_ERR_INVALID_ARG.
 */
lapl_status lapl_attn_set_fault_injection(lapl_attn_handle h, unsigned long long wait_ns,
                                          int skip_last_copy);

/* Launch choices of a plan (fixed at create). */
typedef struct {
  int cdist_tma;      /* 3 (Gaussian kernel only): the squared distances are formed as
                         |x|^2 + |l|^2 - 2 x.l with x.l on the tensor cores (TF32 high/low
                         split, fp32 accumulation; bit for bit the direct sum on integer
                         inputs, to rounding otherwise); 2: the distance kernel's token chunks
                         are loaded by the Tensor Memory Accelerator and half of each warp's
                         landmarks take the q + l - 2 min(q, l) form on the ALU pipe (same
                         distances bit for bit on integer inputs, to rounding otherwise); 1:
                         TMA-fed, every term as |q - l|; 0: cp.async-fed, every term as
                         |q - l| (or (q - l)^2).  1 and 0 give the same distances bit for
                         bit.                                                               */
  int cdist_ctas;     /* persistent CTAs of the distance kernel                              */
  int cdist_threads;  /* threads per distance-kernel CTA                                     */
  int ns_cluster;     /* CTAs per head in the Newton-Schulz solve: 1, or 2 (a cluster pair,
                         m > 32, on request); same X bit for bit                            */
  int ns_tensor_core; /* 1: the solve's products run on the tensor cores (TF32 high/low
                         split, fp32 accumulation); X agrees to rounding                     */
  int ns_exclusive;   /* 1: the solve is the longer chain and runs first, on the launching
                         stream, with SMs to itself; 0: the distance kernel is               */
  int bv_splits;      /* CTAs per head of the B V kernel                                     */
  int bv_tensor_core; /* 1: B V on the tensor cores (TF32 high/low split, fp32 accumulation;
                         d a multiple of 16, N a multiple of 4); 0: CUDA-core FMA tiles     */
  int out_tensor_core; /* 1: O = A^ M on the tensor cores (TF32 high/low split, fp32
                         accumulation; d a multiple of 16 and <= 64, N a multiple of 4);
                         0: CUDA-core FMA tiles                                             */
} lapl_attn_plan_info;

/*
 * Fill *info.  Choices made at create: for the Laplacian kernel with fp32 inputs and d = 32 or
 * 64 the split-pipe TMA kernel (cdist_tma = 2; two CTAs per SM, one CTA of twice the warps for
 * m = 64), cp.async otherwise; for the Gaussian
 * kernel with d = 32 or 64 the tensor-core kernel (cdist_tma = 3), cp.async otherwise; for the
 * solve one CTA per head, with tensor-core products for m >= 25 and
 * CUDA-core products for m <= 16.  Environment variables read at create override them:
 * LAPL_ATTN_CDIST_FEED = "cp.async" (always), "tma" (wherever the plain TMA kernel exists: fp32
 * with d = 32 or 64, bf16 with d = 64) or "l1" (the split-pipe kernel, where it exists), both
 * only with B*H*N >= 128; LAPL_ATTN_NS_KERNEL = "ffma", "pair" (a CTA pair per head, m > 32) or
 * "tc" (tensor-core products).
 */
lapl_status lapl_attn_plan_info_get(lapl_attn_handle h, lapl_attn_plan_info* info);

/*
 * Forward pass for callers that cannot allocate device memory (for example code embedded in a
 * host application that owns every allocation, or a plugin that must not call cudaMalloc).
 * The paper has no counterpart: this is a deployment convenience of this library.
 *
 * Same inputs, outputs and results as lapl_attn_forward (bit for bit), but no workspace
 * argument: the workspace lives in a 32 MiB array in the library's own device memory, which
 * every GPU that loads the library holds until the process exits.  Only the part of the
 * workspace a plain forward uses is placed there (not the regions lapl_attn_forward_train keeps
 * for the backward pass).  It fits the stage-1 vision shape (B=8, H=2, 56x56 tokens, d=32,
 * m=49: about 23 MB) and smaller problems; larger ones (the 28x28, B=32, H=4 shape already
 * needs 42 MB) are rejected with LAPL_ERR_WORKSPACE and a message in lapl_attn_last_error()
 * that states the bytes needed.  Allocates nothing.
 *
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current and keeps it for the life of the process; make that first call before
 * any stream capture, and do not use this entry point on a device after cudaDeviceReset.  All
 * calls share the one array: calls that may overlap on the GPU (other streams, other handles,
 * other threads) race on it and must be serialised by the caller.  Every region the forward
 * uses is written before it is read, so nothing needs clearing between calls.
 */
lapl_status lapl_attn_forward_noalloc(lapl_attn_handle h, const void* q, const void* k,
                                      const void* v, const float* bias, void* out, void* stream);

/*
 * Backward pass: the gradients of a loss with dLoss/dO = dout through the whole forward (the
 * pages claim forward and backward CUDA kernels: English page, 2 "CUDA Acceleration"; German
 * page, 2; they give no gradient, so it is the chain rule through every forward step).
 *
 *   q, k, v, bias   the forward's inputs (bias NULL = zeros), unchanged since that forward;
 *   dout            device [B,H,N,d] fp32, dLoss/dO;
 *   dq, dk, dv      device [B,H,N,d] fp32, written (fp32 also for bf16 inputs);
 *   dbias           device [H,m] fp32 or NULL: written with the sum over the batch of
 *                   dLoss/dbias (zeros when whiten = 0);
 *   fwd_workspace   the workspace of that forward, which must have been
 *                   lapl_attn_forward_train on the same handle, untouched since: the backward
 *                   reads the landmarks, the Newton-Schulz iterates, A, B, the column
 *                   statistics, the B V partials and M from it;
 *   bwd_workspace   device, >= lapl_attn_backward_workspace_size bytes, overwritten.
 * Derivative conventions: d|x - y|/dx = sgn(x - y) with sgn(0) = 0 (for the Gaussian kernel
 * 2 (x - y)); the norms of X0 = W^T / (|W|_1 |W|_inf) differentiate through their first
 * maximal column / row.  Stream-ordered, asynchronous, no allocation; 7 launches.
 * LAPL_ERR_UNSUPPORTED with the CG solver.  Other errors as for forward().
 */
lapl_status lapl_attn_backward_workspace_size(lapl_attn_handle h, size_t* bytes);
lapl_status lapl_attn_backward(lapl_attn_handle h, const void* q, const void* k, const void* v,
                               const float* bias, const float* dout, float* dq, float* dk,
                               float* dv, float* dbias, const void* fwd_workspace,
                               size_t fwd_workspace_bytes, void* bwd_workspace,
                               size_t bwd_workspace_bytes, void* stream);
/* Number of kernels one backward launches: 8 (0 with the CG solver or an empty batch). */
int lapl_attn_backward_kernels(lapl_attn_handle h);

/* Release the plan (host state only).  NULL is accepted. */
lapl_status lapl_attn_destroy(lapl_attn_handle h);

#ifdef __cplusplus
}
#endif

#endif /* LAPL_ATTN_H */
