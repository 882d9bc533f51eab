// C-ABI entry points of libssmscan.so: host-side validation, path selection and launch.
// Every argument problem is found here, before anything is enqueued.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "internal.h"
#include "ssmscan.h"

namespace ssm {
static std::atomic<uint64_t> g_launches{0};
void note_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
}  // namespace ssm

namespace {

thread_local char g_last_error[512] = "";

ssm_status_t fail(ssm_status_t s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return s;
}

ssm_status_t ok() {
    g_last_error[0] = '\0';
    return SSM_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// A strided view of `sizes` may not use negative strides.
bool strides_nonneg(const int64_t* st, int nd) {
    for (int i = 0; i < nd; ++i)
        if (st[i] < 0) return false;
    return true;
}

// Sufficient condition for a view to have no two index tuples at one address: sorted by
// stride, each dimension of size > 1 steps over everything the smaller ones span.
bool non_overlapping(const int64_t* sizes, const int64_t* st, int nd) {
    int64_t sz[4], sd[4];
    int k = 0;
    for (int i = 0; i < nd; ++i)
        if (sizes[i] > 1) {
            sz[k] = sizes[i];
            sd[k] = st[i];
            ++k;
        }
    for (int i = 0; i < k; ++i)
        for (int j = i + 1; j < k; ++j)
            if (sd[j] < sd[i]) {
                std::swap(sd[i], sd[j]);
                std::swap(sz[i], sz[j]);
            }
    int64_t span = 1;
    for (int i = 0; i < k; ++i) {
        if (sd[i] < span) return false;
        span = sd[i] * sz[i];
    }
    return true;
}

// Byte range [lo, hi) spanned by a strided view with non-negative strides (empty if any size is 0).
struct Span {
    uintptr_t lo = 0, hi = 0;
};

Span span_of(const void* p, const int64_t* sizes, const int64_t* st, int nd, size_t esz) {
    Span r;
    if (!p) return r;
    int64_t ext = 0;
    for (int i = 0; i < nd; ++i) {
        if (sizes[i] <= 0) return r;
        ext += (sizes[i] - 1) * st[i];
    }
    r.lo = reinterpret_cast<uintptr_t>(p);
    r.hi = r.lo + (uintptr_t)(ext * (int64_t)esz + (int64_t)esz);
    return r;
}

Span span_dense(const void* p, int64_t elems, size_t esz) {
    Span r;
    if (!p || elems <= 0) return r;
    r.lo = reinterpret_cast<uintptr_t>(p);
    r.hi = r.lo + (uintptr_t)elems * esz;
    return r;
}

bool overlap(const Span& a, const Span& b) { return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi; }

constexpr int64_t kMaxDState = 256;
constexpr int kMaxPhaseEvents = 64;
constexpr int kMaxConvWidth = 4;

ssm_status_t validate_scan(const ssm_scan_params* p, ssm::ScanArgs* out) {
    if (!p) return fail(SSM_ERR_INVALID_ARG, "params is NULL");
    if (p->batch < 1 || p->dim < 1 || p->seqlen < 0)
        return fail(SSM_ERR_INVALID_ARG, "need batch >= 1, dim >= 1, seqlen >= 0 (got %lld, %lld, %lld)",
                    (long long)p->batch, (long long)p->dim, (long long)p->seqlen);
    if (p->dstate < 1) return fail(SSM_ERR_INVALID_ARG, "dstate must be >= 1");
    if (p->dstate > kMaxDState)
        return fail(SSM_ERR_UNSUPPORTED, "dstate %lld > %lld", (long long)p->dstate, (long long)kMaxDState);
    if (p->io_dtype != SSM_DTYPE_F32 && p->io_dtype != SSM_DTYPE_BF16)
        return fail(SSM_ERR_INVALID_ARG, "io_dtype %d unknown", p->io_dtype);
    if (p->discretization != SSM_DISC_DELTA_B && p->discretization != SSM_DISC_ZOH)
        return fail(SSM_ERR_INVALID_ARG, "discretization %d unknown", p->discretization);
    if ((p->delta_softplus != 0 && p->delta_softplus != 1) || (p->reverse != 0 && p->reverse != 1))
        return fail(SSM_ERR_INVALID_ARG, "delta_softplus and reverse must be 0 or 1");
    if (p->chunk_len < 0) return fail(SSM_ERR_INVALID_ARG, "chunk_len must be >= 0");
    if (p->reserved != 0 || p->reserved2 != 0 || (p->debug_flags & ~SSM_DEBUG_SKIP_FIRST_LOAD) != 0)
        return fail(SSM_ERR_INVALID_ARG, "unknown debug_flags or nonzero reserved field");
    if (p->algorithm != SSM_SCAN_ALGO_SERIAL && p->algorithm != SSM_SCAN_ALGO_ASSOC)
        return fail(SSM_ERR_INVALID_ARG, "algorithm %d unknown", p->algorithm);
    if (p->algorithm == SSM_SCAN_ALGO_ASSOC &&
        (p->reverse || p->discretization != SSM_DISC_DELTA_B || p->conv_weight || (p->dstate != 16 && p->dstate != 32)))
        return fail(SSM_ERR_UNSUPPORTED,
                    "the associative scan takes N = 16 or 32, forward, delta B, no conv prologue");
    if (p->n_phase_events < 0 || p->n_phase_events > kMaxPhaseEvents || (p->n_phase_events > 0) != (p->phase_events != nullptr))
        return fail(SSM_ERR_INVALID_ARG, "phase_events must be NULL with n_phase_events == 0, or hold 1..%d events",
                    kMaxPhaseEvents);
    if (!p->A) return fail(SSM_ERR_INVALID_ARG, "A is NULL");
    if (p->conv_weight) {
        if (p->conv_width < 1 || p->conv_width > kMaxConvWidth)
            return fail(SSM_ERR_INVALID_ARG, "conv_width must be 1..%d (got %d)", kMaxConvWidth, p->conv_width);
        if (p->reverse) return fail(SSM_ERR_UNSUPPORTED, "the conv1d prologue runs forward only");
        if (!aligned(p->conv_weight, 4) || (p->conv_bias && !aligned(p->conv_bias, 4)))
            return fail(SSM_ERR_INVALID_ARG, "conv_weight and conv_bias must be 4-byte aligned");
    }
    if (p->seqlen > 0 && (!p->x || !p->delta || !p->B || !p->C || !p->y))
        return fail(SSM_ERR_INVALID_ARG, "x, delta, B, C and y are required");
    const size_t esz = p->io_dtype == SSM_DTYPE_BF16 ? 2 : 4;
    const void* io[] = {p->x, p->delta, p->B, p->C, p->z, p->y, p->conv_weight ? p->conv_x_prev : nullptr};
    for (const void* q : io)
        if (q && !aligned(q, esz)) return fail(SSM_ERR_INVALID_ARG, "I/O pointer not aligned to its dtype");
    const void* f32[] = {p->A, p->D, p->delta_bias, p->h0, p->h_last};
    for (const void* q : f32)
        if (q && !aligned(q, 4)) return fail(SSM_ERR_INVALID_ARG, "fp32 pointer not 4-byte aligned");
    const int64_t* strides[] = {p->x_stride, p->delta_stride, p->z_stride, p->y_stride, p->B_stride, p->C_stride};
    for (const int64_t* s : strides)
        if (!strides_nonneg(s, 3)) return fail(SSM_ERR_INVALID_ARG, "negative stride");
    const int64_t ysz[3] = {p->batch, p->seqlen, p->dim};
    if (p->seqlen > 0 && !non_overlapping(ysz, p->y_stride, 3))
        return fail(SSM_ERR_INVALID_ARG, "y strides overlap");
    const int64_t state_elems = p->batch * p->dim * p->dstate;
    if (p->h_last && p->h0 && p->h_last != p->h0 &&
        overlap(span_dense(p->h0, state_elems, 4), span_dense(p->h_last, state_elems, 4)))
        return fail(SSM_ERR_INVALID_ARG, "h0 and h_last partly overlap");
    if (p->seqlen > 0) {
        // y and h_last are written while every input is still being read: their memory may
        // not overlap any input (h_last may be h0 itself, which is read before it is written)
        const int64_t act[3] = {p->batch, p->seqlen, p->dim};
        const int64_t bc[3] = {p->batch, p->seqlen, p->dstate};
        const Span ys = span_of(p->y, act, p->y_stride, 3, esz);
        const Span hs = span_dense(p->h_last, state_elems, 4);
        const int K = p->conv_weight ? p->conv_width : 0;
        const Span ins[] = {span_of(p->x, act, p->x_stride, 3, esz),
                            span_of(p->delta, act, p->delta_stride, 3, esz),
                            span_of(p->z, act, p->z_stride, 3, esz),
                            span_of(p->B, bc, p->B_stride, 3, esz),
                            span_of(p->C, bc, p->C_stride, 3, esz),
                            span_dense(p->A, p->dim * p->dstate, 4),
                            span_dense(p->D, p->dim, 4),
                            span_dense(p->delta_bias, p->dim, 4),
                            span_dense(p->h0 != p->h_last ? p->h0 : nullptr, state_elems, 4),
                            span_dense(p->conv_weight, p->dim * K, 4),
                            span_dense(p->conv_weight ? p->conv_bias : nullptr, p->dim, 4),
                            span_dense(p->conv_weight ? p->conv_x_prev : nullptr, p->batch * (K - 1) * p->dim, esz)};
        for (const Span& in : ins)
            if (overlap(ys, in) || overlap(hs, in))
                return fail(SSM_ERR_INVALID_ARG, "y or h_last overlaps an input");
        if (overlap(ys, hs)) return fail(SSM_ERR_INVALID_ARG, "y and h_last overlap");
    }
    ssm::ScanArgs& a = *out;
    a.batch = p->batch;
    a.seqlen = p->seqlen;
    a.dim = p->dim;
    a.dstate = (int)p->dstate;
    a.io_bf16 = p->io_dtype == SSM_DTYPE_BF16;
    a.softplus = p->delta_softplus;
    a.reverse = p->reverse;
    a.zoh = p->discretization == SSM_DISC_ZOH;
    a.x = p->x;
    a.delta = p->delta;
    a.B = p->B;
    a.C = p->C;
    a.z = p->z;
    a.A = p->A;
    a.D = p->D;
    a.bias = p->delta_bias;
    a.h0 = p->h0;
    a.y = p->y;
    a.h_last = p->h_last;
    for (int i = 0; i < 3; ++i) {
        a.xs[i] = p->x_stride[i];
        a.ds[i] = p->delta_stride[i];
        a.zs[i] = p->z_stride[i];
        a.ys[i] = p->y_stride[i];
        a.Bs[i] = p->B_stride[i];
        a.Cs[i] = p->C_stride[i];
    }
    a.chunk_len = p->chunk_len;
    a.workspace = p->workspace;
    a.workspace_bytes = p->workspace_bytes;
    a.debug_flags = p->debug_flags;
    a.algorithm = p->algorithm;
    a.conv_w = p->conv_weight;
    a.conv_b = p->conv_weight ? p->conv_bias : nullptr;
    a.conv_prev = p->conv_weight ? p->conv_x_prev : nullptr;
    a.conv_k = p->conv_weight ? p->conv_width : 0;
    a.status = nullptr;
    a.phase_events = p->phase_events;
    a.n_phase_events = p->n_phase_events;
    auto ext = [](const int64_t* sizes, const int64_t* st) {
        int64_t e = 1;
        for (int i = 0; i < 3; ++i) e += (sizes[i] - 1) * st[i];
        return e;
    };
    const int64_t act[3] = {p->batch, p->seqlen > 0 ? p->seqlen : 1, p->dim};
    const int64_t bc[3] = {p->batch, p->seqlen > 0 ? p->seqlen : 1, p->dstate};
    a.ext_x = ext(act, p->x_stride);
    a.ext_delta = ext(act, p->delta_stride);
    a.ext_z = ext(act, p->z_stride);
    a.ext_y = ext(act, p->y_stride);
    a.ext_B = ext(bc, p->B_stride);
    a.ext_C = ext(bc, p->C_stride);
    if (a.algorithm == SSM_SCAN_ALGO_ASSOC && a.seqlen > 0 && !ssm::scan_fast_supported(a))
        return fail(SSM_ERR_UNSUPPORTED, "the associative scan needs the TMA layout (dense channel-contiguous "
                                         "rows, 16-byte aligned) and a driver");
    return SSM_OK;
}

ssm_status_t validate_conv1d(const ssm_conv1d_params* p, ssm::Conv1dArgs* out) {
    if (!p) return fail(SSM_ERR_INVALID_ARG, "params is NULL");
    if (p->batch < 1 || p->dim < 1 || p->seqlen < 0)
        return fail(SSM_ERR_INVALID_ARG, "need batch >= 1, dim >= 1, seqlen >= 0");
    if (p->width < 1 || p->width > kMaxConvWidth)
        return fail(SSM_ERR_INVALID_ARG, "width must be 1..%d (got %d)", kMaxConvWidth, p->width);
    if (p->io_dtype != SSM_DTYPE_F32 && p->io_dtype != SSM_DTYPE_BF16)
        return fail(SSM_ERR_INVALID_ARG, "io_dtype %d unknown", p->io_dtype);
    if ((p->silu != 0 && p->silu != 1) || p->reserved != 0)
        return fail(SSM_ERR_INVALID_ARG, "silu must be 0 or 1 and reserved 0");
    if (!p->weight) return fail(SSM_ERR_INVALID_ARG, "weight is NULL");
    if (p->seqlen > 0 && (!p->x || !p->y)) return fail(SSM_ERR_INVALID_ARG, "x and y are required");
    const size_t esz = p->io_dtype == SSM_DTYPE_BF16 ? 2 : 4;
    if ((p->dim * (int64_t)esz) % 16 != 0)
        return fail(SSM_ERR_UNSUPPORTED, "dim * element size must be a multiple of 16 bytes");
    const void* io[] = {p->x, p->x_prev, p->y};
    for (const void* q : io)
        if (q && !aligned(q, 16)) return fail(SSM_ERR_INVALID_ARG, "x, x_prev and y must be 16-byte aligned");
    if (!aligned(p->weight, 4) || (p->bias && !aligned(p->bias, 4)))
        return fail(SSM_ERR_INVALID_ARG, "weight and bias must be 4-byte aligned");
    if (p->seqlen > 0) {
        const char* y0 = static_cast<const char*>(p->y);
        const int64_t ybytes = p->batch * p->seqlen * p->dim * (int64_t)esz;
        auto overlaps = [&](const void* q, int64_t bytes) {
            const char* q0 = static_cast<const char*>(q);
            return q && q0 < y0 + ybytes && y0 < q0 + bytes;
        };
        if (overlaps(p->x, ybytes) || overlaps(p->x_prev, p->batch * (p->width - 1) * p->dim * (int64_t)esz))
            return fail(SSM_ERR_INVALID_ARG, "y overlaps x or x_prev");
    }
    ssm::Conv1dArgs& a = *out;
    a.batch = p->batch;
    a.seqlen = p->seqlen;
    a.dim = p->dim;
    a.k = p->width;
    a.io_bf16 = p->io_dtype == SSM_DTYPE_BF16;
    a.silu = p->silu;
    a.x = p->x;
    a.w = p->weight;
    a.bias = p->bias;
    a.x_prev = p->x_prev;
    a.y = p->y;
    a.status = nullptr;
    return SSM_OK;
}

// Sequences this short (a decode step is L = 1) take the short-sequence kernel (or the generic
// one for layouts it does not take): one launch, no TMA tile set-up, the state read once and
// written once (in place when h0 == h_last).
constexpr int64_t kShortSeq = 4;

// Whether every path needs the status header: in the debug build every kernel can report a
// failed index check there.
#ifdef SSM_DEBUG_CHECKS
constexpr bool kStatusEverywhere = true;
#else
constexpr bool kStatusEverywhere = false;
#endif

// The TMA kernels wait (bounded) on their copies, so they need the status header; the split
// sequence adds its chunk carries after it. The short-sequence and generic kernels need none
// (except in the debug build).
bool takes_tma_path(const ssm::ScanArgs& a) {
    if (a.algorithm == SSM_SCAN_ALGO_ASSOC) return a.seqlen > 0;   // validated: TMA layout
    return a.seqlen > kShortSeq && ssm::scan_fast_supported(a);
}

size_t scan_workspace_bytes(const ssm::ScanArgs& a) {
    if (!takes_tma_path(a))
        return kStatusEverywhere && a.seqlen > 0 ? SSM_WORKSPACE_HEADER_BYTES : 0;
    return SSM_WORKSPACE_HEADER_BYTES + ssm::scan_fast_workspace_bytes(a);
}

ssm_status_t cuda_fail(cudaError_t e) {
    return fail(SSM_ERR_CUDA, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
}

ssm_status_t validate_ssd(const ssd_scan_params* p, ssm::SSDArgs* out) {
    if (!p) return fail(SSM_ERR_INVALID_ARG, "params is NULL");
    if (p->batch < 1 || p->seqlen < 0 || p->nheads < 1 || p->headdim < 1 || p->dstate < 1 || p->ngroups < 1)
        return fail(SSM_ERR_INVALID_ARG, "need batch, nheads, headdim, dstate, ngroups >= 1 and seqlen >= 0");
    if (p->nheads % p->ngroups != 0) return fail(SSM_ERR_INVALID_ARG, "ngroups must divide nheads");
    if (p->chunk_size < 1) return fail(SSM_ERR_INVALID_ARG, "chunk_size must be >= 1");
    if (p->io_dtype != SSM_DTYPE_F32 && p->io_dtype != SSM_DTYPE_BF16)
        return fail(SSM_ERR_INVALID_ARG, "io_dtype %d unknown", p->io_dtype);
    if (p->delta_softplus != 0 && p->delta_softplus != 1)
        return fail(SSM_ERR_INVALID_ARG, "delta_softplus must be 0 or 1");
    if (!p->A) return fail(SSM_ERR_INVALID_ARG, "A is NULL");
    if (p->seqlen > 0 && (!p->x || !p->delta || !p->B || !p->C || !p->y))
        return fail(SSM_ERR_INVALID_ARG, "x, delta, B, C and y are required");
    if (p->headdim > 256 || p->dstate > 256)
        return fail(SSM_ERR_UNSUPPORTED, "headdim and dstate must be <= 256");
    const int64_t J = 256 / p->headdim;
    if ((p->dstate + J - 1) / J > 64)
        return fail(SSM_ERR_UNSUPPORTED, "dstate %lld too large for headdim %lld", (long long)p->dstate,
                    (long long)p->headdim);
    const size_t esz = p->io_dtype == SSM_DTYPE_BF16 ? 2 : 4;
    const void* io[] = {p->x, p->delta, p->B, p->C, p->z, p->y};
    for (const void* q : io)
        if (q && !aligned(q, esz)) return fail(SSM_ERR_INVALID_ARG, "I/O pointer not aligned to its dtype");
    const void* f32[] = {p->A, p->D, p->delta_bias, p->h0, p->h_last};
    for (const void* q : f32)
        if (q && !aligned(q, 4)) return fail(SSM_ERR_INVALID_ARG, "fp32 pointer not 4-byte aligned");
    ssm::SSDArgs& a = *out;
    a.batch = p->batch;
    a.seqlen = p->seqlen;
    a.nheads = p->nheads;
    a.headdim = p->headdim;
    a.dstate = p->dstate;
    a.ngroups = p->ngroups;
    a.chunk = p->chunk_size;
    a.io_bf16 = p->io_dtype == SSM_DTYPE_BF16;
    a.softplus = p->delta_softplus;
    a.x = p->x;
    a.delta = p->delta;
    a.A = p->A;
    a.B = p->B;
    a.C = p->C;
    a.D = p->D;
    a.z = p->z;
    a.bias = p->delta_bias;
    a.h0 = p->h0;
    a.y = p->y;
    a.h_last = p->h_last;
    a.workspace = p->workspace;
    a.workspace_bytes = p->workspace_bytes;
    a.status = nullptr;
    return SSM_OK;
}

// Check a workspace of `need` bytes (need > 0) and point `status` at its header.
ssm_status_t attach_workspace(void* ws, size_t bytes, size_t need, unsigned** status) {
    if (!ws || bytes < need || !aligned(ws, 256))
        return fail(SSM_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned", need);
    *status = static_cast<unsigned*>(ws);
    return SSM_OK;
}

}  // namespace

namespace ssm {
// Record a reason for ssm_last_error() on the calling thread and return `s` (for entry points
// defined in other files of the library).
ssm_status_t set_error(ssm_status_t s, const char* msg) { return fail(s, "%s", msg); }

cudaError_t record_phase(const ScanArgs& a, int k, bool last, cudaStream_t st) {
    if (!a.phase_events) return cudaSuccess;
    const int hi = last ? a.n_phase_events : std::min(k + 1, a.n_phase_events);
    for (int i = k; i < hi; ++i) {
        const cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(a.phase_events[i]), st);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}
}  // namespace ssm

extern "C" {

size_t ssm_scan_workspace_size(const ssm_scan_params* p) {
    ssm::ScanArgs a;
    if (validate_scan(p, &a) != SSM_OK) return (size_t)-1;
    return scan_workspace_bytes(a);
}

ssm_status_t ssm_scan_fwd(const ssm_scan_params* p, void* stream) {
    ssm::ScanArgs a;
    ssm_status_t s = validate_scan(p, &a);
    if (s != SSM_OK) return s;
    const size_t need = scan_workspace_bytes(a);
    if (need > 0) {
        s = attach_workspace(a.workspace, a.workspace_bytes, need, &a.status);
        if (s != SSM_OK) return s;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if ((a.debug_flags & SSM_DEBUG_SKIP_FIRST_LOAD) &&
        (a.seqlen <= kShortSeq || a.seqlen > 16 || !ssm::scan_fast_supported(a)))
        return fail(SSM_ERR_INVALID_ARG, "SSM_DEBUG_SKIP_FIRST_LOAD needs %lld < seqlen <= 16 and the TMA path",
                    (long long)kShortSeq);
    if (takes_tma_path(a)) {
        e = ssm::launch_scan_fast(a, st);   // records its own phase events
    } else {
        e = ssm::record_phase(a, 0, false, st);
        if (e == cudaSuccess) {
            if (a.seqlen == 0) {
                if (a.h_last) {
                    const size_t bytes = (size_t)(a.batch * a.dim * a.dstate) * sizeof(float);
                    e = a.h0 ? (a.h0 == a.h_last
                                    ? cudaSuccess
                                    : cudaMemcpyAsync(a.h_last, a.h0, bytes, cudaMemcpyDeviceToDevice, st))
                             : cudaMemsetAsync(a.h_last, 0, bytes, st);
                }
            } else if (a.seqlen <= kShortSeq && ssm::scan_decode_supported(a)) {
                e = ssm::launch_scan_decode(a, st);
            } else {
                e = ssm::launch_scan_generic(a, st);
            }
        }
        if (e == cudaSuccess) e = ssm::record_phase(a, 1, true, st);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    return ok();
}

size_t ssm_causal_conv1d_workspace_size(const ssm_conv1d_params* p) {
    ssm::Conv1dArgs a;
    if (validate_conv1d(p, &a) != SSM_OK) return (size_t)-1;
    return a.seqlen > 0 ? SSM_WORKSPACE_HEADER_BYTES : 0;
}

ssm_status_t ssm_causal_conv1d_fwd(const ssm_conv1d_params* p, void* stream) {
    ssm::Conv1dArgs a;
    ssm_status_t s = validate_conv1d(p, &a);
    if (s != SSM_OK) return s;
    if (a.seqlen == 0) return ok();
    s = attach_workspace(p->workspace, p->workspace_bytes, SSM_WORKSPACE_HEADER_BYTES, &a.status);
    if (s != SSM_OK) return s;
    cudaError_t e = ssm::launch_conv1d(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return ok();
}

size_t ssd_chunk_scan_workspace_size(const ssd_scan_params* p) {
    ssm::SSDArgs a;
    if (validate_ssd(p, &a) != SSM_OK) return (size_t)-1;
    return a.seqlen > 0 && (kStatusEverywhere || ssm::ssd_tc_supported(a)) ? SSM_WORKSPACE_HEADER_BYTES : 0;
}

ssm_status_t ssd_chunk_scan_fwd(const ssd_scan_params* p, void* stream) {
    ssm::SSDArgs a;
    ssm_status_t s = validate_ssd(p, &a);
    if (s != SSM_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (a.seqlen > 0 && (kStatusEverywhere || ssm::ssd_tc_supported(a))) {
        s = attach_workspace(a.workspace, a.workspace_bytes, SSM_WORKSPACE_HEADER_BYTES, &a.status);
        if (s != SSM_OK) return s;
    }
    if (a.seqlen == 0) {
        if (a.h_last) {
            const size_t bytes = (size_t)(a.batch * a.nheads * a.dstate * a.headdim) * sizeof(float);
            e = a.h0 ? (a.h0 == a.h_last ? cudaSuccess
                                         : cudaMemcpyAsync(a.h_last, a.h0, bytes, cudaMemcpyDeviceToDevice, st))
                     : cudaMemsetAsync(a.h_last, 0, bytes, st);
        }
    } else if (ssm::ssd_tc_supported(a)) {
        e = ssm::launch_ssd_tc(a, st);
    } else {
        e = ssm::launch_ssd_reference(a, st);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    return ok();
}

ssm_status_t ssm_check_status(void* workspace, void* stream, int clear) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void* ws = workspace;
    if (!ws) {
        cudaError_t err = cudaSuccess;
        ws = ssm::noalloc_scratch(&err);
        if (!ws) return cuda_fail(err);
    }
    if (!aligned(ws, 256)) return fail(SSM_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    unsigned word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, ws, sizeof(unsigned), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && clear) e = cudaMemsetAsync(ws, 0, sizeof(unsigned), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e);
    if (word != 0) return fail(static_cast<ssm_status_t>(word), "a kernel latched status %u in this workspace", word);
    return ok();
}

const char* ssm_status_string(ssm_status_t s) {
    switch (s) {
        case SSM_OK: return "SSM_OK";
        case SSM_ERR_INVALID_ARG: return "SSM_ERR_INVALID_ARG";
        case SSM_ERR_UNSUPPORTED: return "SSM_ERR_UNSUPPORTED";
        case SSM_ERR_CUDA: return "SSM_ERR_CUDA";
        case SSM_ERR_TIMEOUT: return "SSM_ERR_TIMEOUT";
        case SSM_ERR_WORKSPACE: return "SSM_ERR_WORKSPACE";
        case SSM_ERR_BOUNDS: return "SSM_ERR_BOUNDS";
    }
    return "SSM_ERR_UNKNOWN";
}

const char* ssm_last_error(void) { return g_last_error; }

int ssm_abi_version(void) { return SSMSCAN_ABI_VERSION; }

uint64_t ssm_kernel_launch_count(void) { return ssm::g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
