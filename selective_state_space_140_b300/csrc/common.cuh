// Internal helpers of libmamba_scan.so (not part of the public ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mamba {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Bit set in the scan's device error word when a bounded wait gives up.
constexpr unsigned int kErrWaitTimeout = 1u;

// ---- element access for the two io types --------------------------------
template <typename T>
struct Io;

template <>
struct Io<float> {
    static constexpr int kVec = 4;  // elements per 16-byte vector
    static __device__ __forceinline__ float load(const float* p) { return __ldg(p); }
    static __device__ __forceinline__ void store(float* p, float v) { *p = v; }
    // element i of a 16-byte vector
    static __device__ __forceinline__ float get(const uint4& v, int i) {
        return __uint_as_float(i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w);
    }
};

template <>
struct Io<__nv_bfloat16> {
    static constexpr int kVec = 8;
    static __device__ __forceinline__ float load(const __nv_bfloat16* p) {
        return __bfloat162float(__ldg(p));
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, float v) {
        *p = __float2bfloat16_rn(v);
    }
    static __device__ __forceinline__ float get(const uint4& v, int i) {
        const unsigned w = (i >> 1) == 0 ? v.x : (i >> 1) == 1 ? v.y : (i >> 1) == 2 ? v.z : v.w;
        return __uint_as_float((i & 1) ? (w & 0xffff0000u) : (w << 16));
    }
};

// ---- special-function unit and packed fp32 arithmetic -----------------------
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

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two fp32 lanes in one 64-bit register (sm_100+ packed f32x2 arithmetic).
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack2(f32x2 v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// ---- the decay Abar = 2^x of the recurrence ---------------------------------
// x = dt * A * log2 e <= 0.  ex2.approx is biased near x = 0 (on B300 its
// results over [-1, 0) average 0.1 to 0.4 ulp low), and a state whose decay is
// within a few 1e-5 of 1 keeps such a bias for its whole memory 1/(1 - Abar),
// where it adds up linearly instead of averaging out like rounding does.  The
// fp32-io kernels (ACC) therefore form Abar for |x| < 1/16 as 1 + (2^x - 1)
// from the Taylor series of e^(v), v = x ln 2, to v^4/4! (the next term is
// below 2e-9), rounded once, so that Abar is unbiased there; beyond 1/16 a
// state forgets within 23 steps and ex2.approx's bias stays below 1e-6.
// kAbarC[k] = (ln 2)^k / k!.
constexpr float kAbarC1 = 0.693147180559945f, kAbarC2 = 0.240226506959101f,
                kAbarC3 = 0.0555041086648216f, kAbarC4 = 0.00961812910762848f;
constexpr float kAbarSmall = 0.0625f;

template <bool ACC>
__device__ __forceinline__ float abar_exp2(float x) {
    if constexpr (ACC) {
        float q = __fmaf_rn(x, kAbarC4, kAbarC3);
        q = __fmaf_rn(x, q, kAbarC2);
        q = __fmaf_rn(x, q, kAbarC1);
        const float s = __fmaf_rn(x, q, 1.f);
        return fabsf(x) < kAbarSmall ? s : ex2_approx(x);
    } else {
        return ex2_approx(x);
    }
}

// The same on a pair (the series in packed f32x2 arithmetic; each lane equals
// abar_exp2's result bit for bit).
template <bool ACC>
__device__ __forceinline__ f32x2 abar_exp2_pair(f32x2 x) {
    float x0, x1;
    unpack2(x, x0, x1);
    if constexpr (ACC) {
        f32x2 q = fma2(x, pack2(kAbarC4, kAbarC4), pack2(kAbarC3, kAbarC3));
        q = fma2(x, q, pack2(kAbarC2, kAbarC2));
        q = fma2(x, q, pack2(kAbarC1, kAbarC1));
        float s0, s1;
        unpack2(fma2(x, q, pack2(1.f, 1.f)), s0, s1);
        return pack2(fabsf(x0) < kAbarSmall ? s0 : ex2_approx(x0),
                     fabsf(x1) < kAbarSmall ? s1 : ex2_approx(x1));
    } else {
        return pack2(ex2_approx(x0), ex2_approx(x1));
    }
}

// ---- pointwise functions --------------------------------------------------
// softplus(x) = log(1 + e^x), accurate version (fp32 io): libdevice expf and
// log1pf; above 20 the correction is below 2e-9 relative and x is returned.
__device__ __forceinline__ float softplus_accurate(float x) {
    return x > 20.f ? x : log1pf(expf(x));
}

// softplus(x) = max(x, 0) + log1p(e^-|x|), on the SFU (bf16 io, whose inputs
// carry 2^-9 relative rounding already).  log1p(e) uses its Taylor series
// e - e^2/2 below e = 2^-7 (truncation below e^3/3, i.e. 2e-5 relative) and
// lg2(1 + e) * ln2 above, where the lg2 result is at least 0.011.
// Written with explicit round-to-nearest operations so that every kernel
// (scalar or packed callers) gets bit-identical results.
__device__ __forceinline__ float softplus_fast(float x) {
    const float e = ex2_approx(__fmul_rn(-fabsf(x), kLog2e));
    const float series = __fmaf_rn(__fmul_rn(-0.5f, e), e, e);
    const float lg = __fmul_rn(lg2_approx(__fadd_rn(1.f, e)), kLn2);
    return __fadd_rn(fmaxf(x, 0.f), e < 0.0078125f ? series : lg);
}

// y * SiLU(z) = (y * z) / (1 + e^-z), on the SFU, in a fixed operation order.
__device__ __forceinline__ float gate_silu(float y, float z) {
    const float den = __fadd_rn(ex2_approx(__fmul_rn(z, -kLog2e)), 1.f);
    return __fmul_rn(__fmul_rn(y, z), rcp_approx(den));
}

// SiLU(z) = z * sigmoid(z) = z / (1 + e^-z), on the SFU.  For z << 0 the
// exponential overflows to +inf and the reciprocal gives 0, so SiLU -> -0.
__device__ __forceinline__ float silu_fast(float z) {
    return z * rcp_approx(1.f + ex2_approx(-z * kLog2e));
}

// ---- mbarrier and bulk-copy (TMA) primitives ------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile(
        "{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(
            smem_addr(bar)),
        "r"(bytes)
        : "memory");
}

// 1-D bulk copy global -> shared, completing `bytes` on `bar`.  Both addresses
// 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Bounded wait for phase `parity` of `bar`.  A copy that never lands must not
// hang the GPU: each poll is a try_wait that suspends the thread until the
// phase completes or kWaitSuspendNs nanoseconds pass (a suspended warp issues
// nothing, so waiting costs the other warps no issue slots); after `limit`
// polls this returns false, the caller records the failure in its error word
// and carries on (its results are then garbage, which the host learns from
// mamba_device_status()).  kWaitLimit polls bound a wait near 1.3 s; after a
// first failure a thread polls only kWaitLimitAfterFailure times per later
// wait, so a broken launch still ends in bounded time.
constexpr uint32_t kWaitSuspendNs = 20000;
constexpr uint32_t kWaitLimit = 1u << 16;
constexpr uint32_t kWaitLimitAfterFailure = 1u << 4;

__device__ __forceinline__ bool mbar_wait_n(uint64_t* bar, uint32_t parity, uint32_t limit) {
    const uint32_t a = smem_addr(bar);
    for (uint32_t i = 0; i < limit; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(ok)
            : "r"(a), "r"(parity), "r"(kWaitSuspendNs)
            : "memory");
        if (ok) return true;
    }
    return false;
}

// Arguments of one forward scan, as validated by the C entry point.
struct ScanArgs {
    const void* u;
    const void* delta;
    const float* A_log;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* delta_bias;
    void* y;
    float* last_state;
    int64_t batch, dim, seqlen;
    int dstate;
    int softplus;
    // mamba_selective_scan_fwd_ex only (nullptr otherwise):
    const float* h0;             // [batch, dim, dstate] state before step 0
    const unsigned char* reset;  // [batch, seqlen]: non-zero starts a new document
};

// A scan split along time into nseg segments of seg_len steps (the last may
// be shorter): a summary pass gives each segment's end state from a zero start
// and the sum of its dt, a carry pass chains them, and the full pass runs
// every segment from the state that enters it.
struct SegArgs {
    int seg_len;    // steps per segment, a multiple of 16
    int nseg;       // segments of the sequence (1: no split)
    int grid_nseg;  // segments covered by one launch (nseg, or nseg - 1 for the summary)
    float* hcarry;  // [batch * dim][nseg][dstate]: slot s = state entering segment s
    float* sdt;     // [batch * dim][nseg - 1]: sum of dt over segment s (+inf: a reset)
};

// Scratch memory the forward scan may use for a split: a caller buffer of
// `bytes` (ptr != nullptr: never allocates) or, with ptr == nullptr and
// may_alloc, stream-ordered memory taken and returned on the launch stream.
struct ScanScratch {
    void* ptr;
    size_t bytes;
    bool may_alloc;
};

struct StateUpdateArgs {
    float* state;
    const void* x;
    const void* dt;
    const float* A_log;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* dt_bias;
    void* out;
    int64_t batch, dim;
    int dstate;
    int softplus;
};

// Arguments of the backward scan (gradients for dout = dLoss/dy).
struct ScanBwdArgs {
    ScanArgs f;          // the forward's inputs (y, last_state unused; h0, reset read by the _ex form only)
    const void* dout;    // [batch, dim, L] io
    void* du;            // [batch, dim, L] io
    void* ddelta;        // [batch, dim, L] io
    void* dz;            // [batch, dim, L] io, when z is given
    float* dA_log;       // [dim, N]
    float* dB;           // [batch, L, N]
    float* dC;           // [batch, L, N]
    float* dD;           // [dim] or nullptr
    float* ddelta_bias;  // [dim] or nullptr
    const float* dlast = nullptr;  // [batch, dim, N] gradient on the final state, or nullptr (_ex only)
};

// Launchers (return the cudaError_t of the launch).
// cudaErrorMemoryAllocation: the split needs more than a caller buffer holds.
cudaError_t launch_scan_fwd(const ScanArgs& a, bool bf16, cudaStream_t stream,
                            const ScanScratch& scratch);
// Synchronise `stream`, then read and clear the scan's device error word.
cudaError_t read_and_clear_device_error(unsigned int* word, cudaStream_t stream);
// Read and clear the decode kernels' device error word (after a synchronise).
cudaError_t read_and_clear_decode_error(unsigned int* word);
cudaError_t launch_state_update(const StateUpdateArgs& a, bool bf16, cudaStream_t stream);
// Zeroes the summed gradients, takes stream-ordered checkpoint scratch, runs
// the backward kernel and returns the scratch, all on `stream`.
cudaError_t launch_scan_bwd(const ScanBwdArgs& a, bool bf16, cudaStream_t stream);

// Complex-state scan: B, C [batch][L][N][2] (re, im); last_state [batch][dim][N][2].
cudaError_t launch_scan_complex(const void* u, const void* delta, const float* A_log_re,
                                const float* A_im, const void* B, const void* C, const float* D,
                                const void* z, const float* delta_bias, bool softplus, void* y,
                                float* last_state, int64_t batch, int64_t dim, int64_t seqlen,
                                int dstate, bool bf16, cudaStream_t stream);

// Causal depthwise conv1d (+ SiLU) over [batch][dim][L] rows; states [batch][dim][width-1].
cudaError_t launch_causal_conv1d(const void* x, const float* w, const float* bias,
                                 const void* st_in, void* out, void* st_out, int64_t batch,
                                 int64_t dim, int64_t L, int width, bool silu, bool bf16,
                                 cudaStream_t stream);
// One token per row; the conv state shifts in place.
cudaError_t launch_conv1d_update(void* state, const void* x, const float* w, const float* bias,
                                 void* out, int64_t batch, int64_t dim, int width, bool silu,
                                 bool bf16, cudaStream_t stream);
// Test hook: a wait that never completes, given up after `limit` polls.
cudaError_t launch_bounded_wait_probe(uint32_t limit, cudaStream_t stream);

}  // namespace mamba
