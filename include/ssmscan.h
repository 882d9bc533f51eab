/*
 * ssmscan.h — C ABI of libssmscan.so: the selective-scan (Mamba) and SSD (Mamba-2)
 * forward passes on one NVIDIA B300 (sm_103a).
 *
 * Conventions for every entry point
 *  - Pointers in the params structs are DEVICE pointers owned by the caller; the library
 *    never allocates, frees or keeps them after the call returns.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream). Work is
 *    enqueued on it and the call returns without synchronising (except ssm_check_status).
 *  - Argument errors are detected on the host before anything is launched and return
 *    SSM_ERR_INVALID_ARG (shape, stride, pointer, dtype or alignment problem) or
 *    SSM_ERR_UNSUPPORTED (a valid request this library does not implement); a one-line
 *    reason is then available from ssm_last_error() on the calling thread.
 *  - A failed launch returns SSM_ERR_CUDA; the CUDA error string is in ssm_last_error().
 *  - Device-side failures are reported in the caller's workspace: its first
 *    SSM_WORKSPACE_HEADER_BYTES hold a status word that kernels with bounded waits set when a
 *    wait gives up, and ssm_check_status() reads it. A workspace must start with that header
 *    zeroed (cudaMemset once before its first use); ssm_check_status(..., clear = 1) zeroes it
 *    again. Calls that need no workspace (ssm_*_workspace_size() == 0) run kernels with no
 *    device-side waits and have nothing to report.
 *  - Thread-safe. Calls on different streams may run concurrently as long as their output and
 *    workspace buffers do not overlap. The library keeps no state between calls besides the
 *    calling thread's last-error string, a process-wide count of launched kernels, and the
 *    fixed scratch buffer of ssm_scan_fwd_noalloc (see there).
 *  - Arithmetic: inputs in the I/O dtype (fp32 or bf16) are widened to fp32; the state and
 *    every intermediate are fp32; y is rounded to the I/O dtype (round to nearest even).
 *
 * Notation follows the pages: b batch, L sequence length, D channels (d_inner), N state
 * size (d_state); for SSD H heads, P head dimension, G groups of (B, C), Q chunk length.
 */
#ifndef SSMSCAN_H
#define SSMSCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SSMSCAN_ABI_VERSION 4

/* Bytes at the start of every workspace that hold the device status word (a uint32 at offset 0;
 * the rest is reserved). */

/* The debug build of the library (libssmscan_debug.so, built with -DSSM_DEBUG_CHECKS) checks every
 * index its kernels compute for global memory against the array it addresses; a failed check
 * latches SSM_ERR_BOUNDS in the call's status word and skips the access. In that build every
 * call with L > 0 needs a workspace of at least SSM_WORKSPACE_HEADER_BYTES (the *_workspace_size
 * queries say so). Results are otherwise identical to the normal build's. */
#define SSM_WORKSPACE_HEADER_BYTES 256

#if defined(__GNUC__)
#define SSMSCAN_API __attribute__((visibility("default")))
#else
#define SSMSCAN_API
#endif

typedef enum {
    SSM_OK = 0,
    SSM_ERR_INVALID_ARG = 1,
    SSM_ERR_UNSUPPORTED = 2,
    SSM_ERR_CUDA = 3,
    SSM_ERR_TIMEOUT = 4,   /* a bounded device-side wait gave up (see ssm_check_status) */
    SSM_ERR_WORKSPACE = 5, /* workspace missing, too small or misaligned */
    SSM_ERR_BOUNDS = 6     /* debug build only: a kernel's index check failed and the access was
                              skipped (see ssm_check_status) */
} ssm_status_t;

typedef enum { SSM_DTYPE_F32 = 0, SSM_DTYPE_BF16 = 1 } ssm_dtype_t;

/* How B_bar x is formed from delta, A and B.
 * SSM_DISC_DELTA_B: B_bar x = delta * B * x, the simplified discretisation of every
 *   selective listing on the pages ("Mamba/SSM complete guide" section 5 `selective_scan`,
 *   einsum "bld,bln,bld->bldn"; "State Space Model / Mamba", "Mamba風の選択的SSMの実装").
 * SSM_DISC_ZOH: exact zero-order hold for diagonal A, B_bar = (exp(delta a) - 1) / a * B
 *   ("State Space Model / Mamba", "Zero-Order Hold" and `discretize_zoh`; "Mamba/SSM
 *   complete guide" section 2 ZOH formula), with the limit delta * B where a == 0. */
typedef enum { SSM_DISC_DELTA_B = 0, SSM_DISC_ZOH = 1 } ssm_discretization_t;

/* How the recurrence walks the sequence inside a chunk (ssm_scan_params.algorithm); both give
 * the same result up to fp32 rounding.
 *  SSM_SCAN_ALGO_SERIAL (default): each lane walks its states' steps one after the other.
 *  SSM_SCAN_ALGO_ASSOC: each warp runs an inclusive scan of the (A_bar, B_bar x) pairs of a
 *    32-step tile over its lanes with the operator (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2)
 *    ("Mamba/SSM complete guide" section 5 `parallel_scan`), tiles joined through the state.
 *    About ten times slower on B300 (eleven shuffles per state and step); N = 16 or 32,
 *    forward, delta B, no conv prologue, and the TMA layout (dense channel-contiguous rows,
 *    16-byte aligned); anything else is SSM_ERR_UNSUPPORTED. */
typedef enum { SSM_SCAN_ALGO_SERIAL = 0, SSM_SCAN_ALGO_ASSOC = 1 } ssm_scan_algo_t;

/* Test hooks (debug_flags). SSM_DEBUG_SKIP_FIRST_LOAD: the TMA path never issues the copy
 * of its first tile, so its bounded wait runs out (about one second), the kernel latches
 * SSM_ERR_TIMEOUT in the workspace's status word and returns with nothing in flight. Accepted
 * only when the whole sequence fits in that first tile (5 <= L <= 16) and the TMA path
 * applies; otherwise the call returns SSM_ERR_INVALID_ARG. */
#define SSM_DEBUG_SKIP_FIRST_LOAD 1

/*
 * Mamba-1 selective scan, one independent recurrence per (batch, channel):
 *   dt_t   = softplus(delta[b,t,d] + delta_bias[d])      (softplus(v) = log(1 + e^v))
 *   A_bar  = exp(dt_t * A[d,n])
 *   h[n]   = A_bar * h[n] + dt_t * B[b,t,n] * x[b,t,d]    (or the ZOH form above)
 *   y      = sum_n C[b,t,n] * h[n]  +  D[d] * x[b,t,d]
 *   y     *= silu(z[b,t,d]) = z / (1 + e^-z)
 * The output at t reads the state after x_t has entered it. The state starts at h0
 * (zeros when NULL) and its value after the last step is written to h_last. h_last may be
 * the same buffer as h0 (any L, any chunking: the state is read before it is overwritten);
 * with L = 1 that is the single-token (decode) step that advances a cached state in place
 * ("Mamba/SSM complete guide" section 2: recurrent inference with a constant-size state).
 * Pages: "Mamba/SSM complete guide" section 5, listing `selective_scan` (discretise, loop,
 * readout, u*D) and MambaBlock.forward (y * silu(z)); "論文解説: Mamba" "選択機構"
 * (softplus) and "Hardware-Aware Parallel Scan" (the recurrence, zero initial state).
 *
 * Optional prologue (conv_weight != NULL): x is the raw input of the block's x branch, and
 * the scan runs on u = silu(causal depthwise conv1d(x)) instead, for the input term and the
 * D skip alike (see ssm_causal_conv1d_fwd for the convolution). Forward direction only
 * (reverse with the prologue is SSM_ERR_UNSUPPORTED). The convolved input is not written out.
 */
typedef struct ssm_scan_params {
    int64_t batch;          /* b >= 1 */
    int64_t seqlen;         /* L >= 0 (L == 0: nothing is launched except copying h0 to h_last) */
    int64_t dim;            /* D >= 1 */
    int64_t dstate;         /* N, 1 <= N <= 256 */
    int32_t io_dtype;       /* ssm_dtype_t of x, delta, z, B, C and y */
    int32_t delta_softplus; /* 1: dt = softplus(delta + bias); 0: dt = delta + bias */
    int32_t reverse;        /* 1: run t = L-1 .. 0 (h_last is then the state after t = 0) */
    int32_t discretization; /* ssm_discretization_t */
    const void* x;          /* (b, L, D), strides x_stride */
    const void* delta;      /* (b, L, D), strides delta_stride; a channel stride of 0 gives
                               one delta per token shared by all channels */
    const void* B;          /* (b, L, N), strides B_stride, shared by all channels */
    const void* C;          /* (b, L, N), strides C_stride, shared by all channels */
    const void* z;          /* (b, L, D) or NULL (no gate), strides z_stride */
    const float* A;         /* (D, N) fp32, contiguous; expected <= 0 (not enforced) */
    const float* D;         /* (D) fp32 or NULL (no skip) */
    const float* delta_bias;/* (D) fp32 or NULL (zero bias) */
    const float* h0;        /* (b, D, N) fp32 contiguous, or NULL (zeros) */
    void* y;                /* (b, L, D) in io_dtype, strides y_stride; its memory range must not
                               overlap that of any input (checked) */
    float* h_last;          /* (b, D, N) fp32 contiguous, or NULL (not written) */
    int64_t x_stride[3];    /* element strides for (b, t, d); 0 broadcasts */
    int64_t delta_stride[3];
    int64_t z_stride[3];
    int64_t y_stride[3];    /* y must not broadcast: all strides > 0 unless the size is 1 */
    int64_t B_stride[3];    /* (b, t, n) */
    int64_t C_stride[3];
    int64_t chunk_len;      /* steps per chunk when the sequence is split across CTAs (the TMA
                               path rounds it up to a multiple of 32 and to at least L / 65535;
                               >= L, the reverse direction, or a path that does not split: one
                               chunk); 0 = let the library choose. The result does not depend on
                               it beyond fp32 rounding. With more than one chunk the call needs
                               nchunks * b * D * N * 4 + (nchunks - 1) * b * D * 4 bytes of
                               workspace after the header. */
    void* workspace;        /* device scratch of ssm_scan_workspace_size() bytes, 256-byte
                               aligned, header zeroed before first use (see above); may be NULL
                               when that size is 0 */
    size_t workspace_bytes;
    int32_t debug_flags;    /* 0 in normal use; SSM_DEBUG_* test hooks */
    int32_t reserved;       /* must be 0 */
    const float* conv_weight; /* (D, K) fp32 contiguous, or NULL (no prologue: x enters as is) */
    const float* conv_bias;   /* (D) fp32 or NULL (zero bias) */
    const void* conv_x_prev;  /* (b, K-1, D) in io_dtype, contiguous: the K-1 raw inputs before
                                 x[:, 0] (the tail of the previous segment), or NULL (zeros) */
    int32_t conv_width;       /* K, 1 <= K <= 4, when conv_weight is set; ignored otherwise */
    int32_t reserved2;        /* must be 0 */
    void* const* phase_events;/* NULL, or n_phase_events cudaEvent_t handles (passed as void*) for
                                 timing the call's kernels: events[0] is recorded on the stream
                                 before the first kernel the call launches and events[k] after its
                                 k-th kernel; entries past the last kernel are recorded after it
                                 too (the long-sequence path launches 3 kernels: local pass, chunk
                                 carry, output pass; the others 1) */
    int32_t n_phase_events;   /* entries of phase_events (0 when it is NULL) */
    int32_t algorithm;        /* ssm_scan_algo_t: SSM_SCAN_ALGO_SERIAL (0) unless chosen */
} ssm_scan_params;

/* Bytes of device workspace ssm_scan_fwd needs for these params: 0 for the paths without
 * device-side waits (short sequences, generic layouts), else SSM_WORKSPACE_HEADER_BYTES plus
 * the chunk carries of a split sequence. Host only; its first call may look up a driver entry
 * point (cudaGetDriverEntryPointByVersion), nothing else. Returns (size_t)-1 when the params
 * are invalid. */
SSMSCAN_API size_t ssm_scan_workspace_size(const ssm_scan_params* p);

/* Enqueue the selective scan on `stream`. Returns SSM_OK once launched. */
SSMSCAN_API ssm_status_t ssm_scan_fwd(const ssm_scan_params* p, void* stream);

/*
 * Allocation-free variant of ssm_scan_fwd. The pages have no counterpart: it serves callers
 * that cannot allocate device memory or pass a workspace (for example a host application
 * whose device memory is fixed at start-up, or a plugin inside another runtime that owns all
 * device allocations), and callers that cannot afford cudaMalloc's implicit synchronisation.
 *  - Same arguments and results as ssm_scan_fwd; p->workspace and p->workspace_bytes are
 *    ignored. Inputs and outputs are still the caller's.
 *  - The workspace (status header and the chunk carries of the long-sequence path) comes from
 *    a buffer compiled into the library, SSM_NOALLOC_SCRATCH_BYTES (16 MiB) of device memory
 *    on every GPU that loads the library, held until the process exits (the same value is
 *    returned by ssm_noalloc_scratch_bytes()). A call that needs more
 *    (ssm_scan_workspace_size(p) > SSM_NOALLOC_SCRATCH_BYTES) returns SSM_ERR_UNSUPPORTED
 *    before anything is launched; a larger chunk_len needs less.
 *  - The first call on a device looks up the buffer's device address (cudaGetSymbolAddress)
 *    with that device current; make that first call before any stream capture.
 *  - Every call shares the one buffer, which keeps the last call's contents (the carries need
 *    no zeroing: each call writes every element it later reads; the status header starts at
 *    zero when the library loads and is read and cleared by ssm_check_status(NULL, ...)).
 *    Calls whose work overlaps on the GPU (different streams, or different host threads) race
 *    on it: serialise them.
 *  - It calls no cudaMalloc, cudaFree or other allocating routine.
 */
#define SSM_NOALLOC_SCRATCH_BYTES (16u << 20)
SSMSCAN_API ssm_status_t ssm_scan_fwd_noalloc(const ssm_scan_params* p, void* stream);

/* SSM_NOALLOC_SCRATCH_BYTES of the library that was loaded. */
SSMSCAN_API size_t ssm_noalloc_scratch_bytes(void);

/*
 * Causal depthwise convolution along t with K taps per channel, then optionally SiLU: the
 * prologue of the Mamba block's x branch,
 *   v[b,t,d] = bias[d] + sum_{k=0}^{K-1} weight[d,k] * xp[b, t+k, d],   y = silu(v) or v,
 * where xp is x preceded by the K-1 inputs x_prev (zeros when NULL): weight[d, K-1] multiplies
 * x_t and weight[d, 0] multiplies x_{t-K+1}. This is a convolution layer with groups = D,
 * kernel K and padding K-1 whose output is cut to the first L steps.
 * Pages: "Mamba/SSM complete guide" section 5 `MambaBlock` (nn.Conv1d(d_inner, d_inner,
 * d_conv, groups = d_inner, padding = d_conv - 1), output [:, :, :L], then F.silu);
 * "論文解説: Mamba" "Mambaブロックの全体構成" (a d_conv = 4 convolution, then SiLU).
 * All tensors dense and contiguous; every pointer 16-byte aligned.
 */
typedef struct ssm_conv1d_params {
    int64_t batch;          /* b >= 1 */
    int64_t seqlen;         /* L >= 0 (0: nothing is launched) */
    int64_t dim;            /* D >= 1; D * element size must be a multiple of 16 bytes */
    int32_t width;          /* K, 1 <= K <= 4 */
    int32_t io_dtype;       /* ssm_dtype_t of x, x_prev and y */
    int32_t silu;           /* 1: y = silu(v); 0: y = v */
    int32_t reserved;       /* must be 0 */
    const void* x;          /* (b, L, D) */
    const float* weight;    /* (D, K) fp32 */
    const float* bias;      /* (D) fp32 or NULL */
    const void* x_prev;     /* (b, K-1, D) or NULL (zeros) */
    void* y;                /* (b, L, D); must not overlap x or x_prev */
    void* workspace;        /* SSM_WORKSPACE_HEADER_BYTES of device memory (the status word of its
                               bounded waits), 256-byte aligned, header zeroed before first use;
                               may be NULL when L == 0 */
    size_t workspace_bytes;
} ssm_conv1d_params;

/* Bytes of device workspace ssm_causal_conv1d_fwd needs (SSM_WORKSPACE_HEADER_BYTES, or 0
 * when L == 0); (size_t)-1 if the params are invalid. */
SSMSCAN_API size_t ssm_causal_conv1d_workspace_size(const ssm_conv1d_params* p);

/* Enqueue the convolution on `stream`. Returns SSM_OK once launched. */
SSMSCAN_API ssm_status_t ssm_causal_conv1d_fwd(const ssm_conv1d_params* p, void* stream);

/*
 * Mamba-2 SSD chunked scan: the same recurrence with one scalar A per head and the state
 * an N x P matrix per (batch, head):
 *   dt_t = softplus(delta[b,t,h] + delta_bias[h]);  S = exp(dt_t A_h) S + dt_t B_t (x) x_t
 *   y_t  = S^T C_t (+ D_h x_t) (* silu(z_t))
 * computed chunk by chunk (Q steps): inside a chunk by matrix products over the masked,
 * decayed C B^T block, across chunks by handing the state on.
 * Pages: "Mamba-2 / Structured State Space Duality" (abeam) "基本アイデア" (semiseparable
 * matrix, block decomposition: diagonal blocks as block products, off-diagonal blocks as a
 * low-rank state hand-off) and "線形形式と二次形式を使い分ける"; "Mamba/SSM complete guide"
 * section 6 "SSD演算の概念" (intra-chunk matrix products, inter-chunk recurrence) and
 * `Mamba2Block` (A per head; B, C of d_state each in in_proj).
 * All tensors are dense and contiguous in the shapes below.
 */
typedef struct ssd_scan_params {
    int64_t batch;          /* b >= 1 */
    int64_t seqlen;         /* L >= 0 */
    int64_t nheads;         /* H >= 1 */
    int64_t headdim;        /* P */
    int64_t dstate;         /* N */
    int64_t ngroups;        /* G >= 1, divides H; head h reads group h / (H / G) */
    int64_t chunk_size;     /* Q >= 1, a hint: the result does not depend on it beyond rounding.
                               The tensor-core kernel (bf16, P = 64, N = 128, 16-byte aligned
                               tensors) always works in 128-step blocks; the CUDA-core kernel
                               in chunks of Q. */
    int32_t io_dtype;       /* ssm_dtype_t of x, delta, B, C, z and y */
    int32_t delta_softplus; /* as for ssm_scan_params */
    const void* x;          /* (b, L, H, P) */
    const void* delta;      /* (b, L, H) */
    const float* A;         /* (H) fp32 */
    const void* B;          /* (b, L, G, N) */
    const void* C;          /* (b, L, G, N) */
    const float* D;         /* (H) fp32 or NULL */
    const void* z;          /* (b, L, H, P) or NULL */
    const float* delta_bias;/* (H) fp32 or NULL */
    const float* h0;        /* (b, H, N, P) fp32 or NULL */
    void* y;                /* (b, L, H, P) in io_dtype */
    float* h_last;          /* (b, H, N, P) fp32 or NULL */
    void* workspace;        /* device scratch of ssd_chunk_scan_workspace_size() bytes, 256-byte
                               aligned, header zeroed before first use; may be NULL when that
                               size is 0 */
    size_t workspace_bytes;
} ssd_scan_params;

/* Bytes of device workspace ssd_chunk_scan_fwd needs: SSM_WORKSPACE_HEADER_BYTES on the
 * tensor-core path (its bounded waits), 0 on the CUDA-core path; (size_t)-1 if invalid. */
SSMSCAN_API size_t ssd_chunk_scan_workspace_size(const ssd_scan_params* p);

/* Enqueue the SSD chunked scan on `stream`. Returns SSM_OK once launched. */
SSMSCAN_API ssm_status_t ssd_chunk_scan_fwd(const ssd_scan_params* p, void* stream);

/* Synchronise `stream`, then return the status word in the header of `workspace` (a device
 * pointer given to earlier calls on this stream): SSM_OK, or SSM_ERR_TIMEOUT if a bounded
 * wait of a kernel that used this workspace gave up since the word was last cleared (that
 * call's outputs are then incomplete), or, in the debug build, SSM_ERR_BOUNDS if a kernel's
 * index check failed. A timeout is visible only through the workspace of
 * the call that had it. workspace == NULL reads the header of the built-in scratch of
 * ssm_scan_fwd_noalloc on the current device. With `clear` != 0 the word is reset to SSM_OK
 * afterwards. Returns SSM_ERR_CUDA if the stream reports an error. */
SSMSCAN_API ssm_status_t ssm_check_status(void* workspace, void* stream, int clear);

/* Static, human-readable name of a status code. */
SSMSCAN_API const char* ssm_status_string(ssm_status_t s);

/* The reason for the last non-OK status returned on the calling thread ("" if none). */
SSMSCAN_API const char* ssm_last_error(void);

/* SSMSCAN_ABI_VERSION of the library that was loaded. */
SSMSCAN_API int ssm_abi_version(void);

/* Number of kernels this library has enqueued in this process so far (all devices,
 * all threads; copies and memsets are not counted). For benchmarks that report how many
 * of the library's kernels ran in a timed region. */
SSMSCAN_API uint64_t ssm_kernel_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* SSMSCAN_H */
