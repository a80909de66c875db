// Single-token decode step (recurrent inference) for sm_103a.
//
// For every (batch, channel) chain: dt = softplus(dt_raw + bias),
// h <- exp(dt*A) h + dt*B*x in place, out = (C.h + D x) * SiLU(z).  Inference
// touches only the previous state (tutorial "核心概念"; mhpn.cn article
// section 3), so the step is bound by reading and writing the fp32 state.
//
// G lanes of one warp share a chain, each owning NPL consecutive states, so a
// warp reads and writes a contiguous run of the state array (one 16-byte
// access per lane when NPL == 4 and the state is 16-byte aligned).  The partial
// sums of C.h are combined with warp shuffles inside the G-lane group.
#include "common.cuh"

namespace mamba {
namespace {

// CPT chains per thread: a warp covers CPT rows of 32 / G consecutive chains
// (contiguous state), and every load of a thread is issued before the first
// use, so that each thread keeps CPT * NPL * 4 bytes of state in flight.
template <typename io_t, int NPL, int G, int CPT, bool VEC>
__global__ void __launch_bounds__(256) state_update_kernel(StateUpdateArgs p) {
    constexpr int CPW = 32 / G;  // chains per warp row
    const int64_t chains = p.batch * p.dim;
    const int lane = threadIdx.x & 31;
    const int g = lane % G;
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
    const int N = p.dstate;

    int64_t chain[CPT];
    bool live[CPT];
    float h[CPT][NPL], A[CPT][NPL], Bv[CPT][NPL], Cv[CPT][NPL], raw[CPT], x[CPT], zv[CPT];
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        chain[c] = (warp * CPT + c) * CPW + lane / G;
        // Whole G-lane groups are live or dead together, so the shuffles below
        // never mix live and dead lanes of one chain.
        live[c] = chain[c] < chains;
        const int64_t ch = live[c] ? chain[c] : 0;
        const int64_t b = ch / p.dim, d = ch % p.dim;
        const float* st = p.state + ch * N + g * NPL;
        const float* al = p.A_log + d * N + g * NPL;
        const io_t* Bb = static_cast<const io_t*>(p.B) + b * N + g * NPL;
        const io_t* Cb = static_cast<const io_t*>(p.C) + b * N + g * NPL;
#pragma unroll
        for (int i = 0; i < NPL; i += 4) {
            if (VEC) {
                const float4 v = *reinterpret_cast<const float4*>(st + i);
                h[c][i] = v.x; h[c][i + 1] = v.y; h[c][i + 2] = v.z; h[c][i + 3] = v.w;
            }
        }
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            const bool ok = VEC || g * NPL + i < N;
            if (!VEC) h[c][i] = ok ? st[i] : 0.f;
            A[c][i] = ok ? __ldg(al + i) : 0.f;
            Bv[c][i] = ok ? Io<io_t>::load(Bb + i) : 0.f;
            Cv[c][i] = ok ? Io<io_t>::load(Cb + i) : 0.f;
        }
        raw[c] = Io<io_t>::load(static_cast<const io_t*>(p.dt) + ch) +
                 (p.dt_bias ? __ldg(p.dt_bias + d) : 0.f);
        x[c] = Io<io_t>::load(static_cast<const io_t*>(p.x) + ch);
        zv[c] = p.z ? Io<io_t>::load(static_cast<const io_t*>(p.z) + ch) : 0.f;
    }

    float acc[CPT];
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        const float dt = !p.softplus ? raw[c]
                         : sizeof(io_t) == 2 ? softplus_fast(raw[c])
                                             : softplus_accurate(raw[c]);
        const float dx = dt * x[c];
        acc[c] = 0.f;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            // A = -exp(A_log) = -2^(A_log * log2 e); Abar = 2^(dt * A * log2 e)
            const float A2 = -ex2_approx(A[c][i] * kLog2e) * kLog2e;
            const float a = ex2_approx(dt * A2);
            h[c][i] = fmaf(a, h[c][i], dx * Bv[c][i]);
            acc[c] = fmaf(Cv[c][i], h[c][i], acc[c]);
        }
    }

#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        if (!live[c]) continue;
        float* st = p.state + chain[c] * N + g * NPL;
        if constexpr (VEC) {
#pragma unroll
            for (int i = 0; i < NPL; i += 4)
                *reinterpret_cast<float4*>(st + i) =
                    make_float4(h[c][i], h[c][i + 1], h[c][i + 2], h[c][i + 3]);
        } else {
#pragma unroll
            for (int i = 0; i < NPL; ++i)
                if (g * NPL + i < N) st[i] = h[c][i];
        }
    }

    const unsigned gmask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (lane / G * G));
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        if (!live[c]) continue;
        float v = acc[c];
#pragma unroll
        for (int off = G / 2; off > 0; off /= 2) v += __shfl_xor_sync(gmask, v, off, G);
        if (g == 0) {
            const int64_t d = chain[c] % p.dim;
            if (p.D) v = fmaf(__ldg(p.D + d), x[c], v);
            if (p.z) v *= silu_fast(zv[c]);
            Io<io_t>::store(static_cast<io_t*>(p.out) + chain[c], v);
        }
    }
}

template <typename io_t, int NPL, int G>
cudaError_t launch(const StateUpdateArgs& a, cudaStream_t stream) {
    const bool vec = (a.dstate % 4 == 0) && (a.dstate == NPL * G) &&
                     (reinterpret_cast<uintptr_t>(a.state) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(a.A_log) % 16 == 0);
    constexpr int CPT = 2;
    const int64_t cpt = vec ? CPT : 1;
    const int64_t warps = (a.batch * a.dim + (32 / G) * cpt - 1) / ((32 / G) * cpt);
    const int64_t blocks = (warps * 32 + 255) / 256;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    if (vec)
        state_update_kernel<io_t, NPL, G, CPT, true><<<unsigned(blocks), 256, 0, stream>>>(a);
    else
        state_update_kernel<io_t, NPL, G, 1, false><<<unsigned(blocks), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

template <typename io_t>
cudaError_t dispatch(const StateUpdateArgs& a, cudaStream_t stream) {
    const int N = a.dstate;
    if (N <= 4) return launch<io_t, 4, 1>(a, stream);
    if (N <= 8) return launch<io_t, 4, 2>(a, stream);
    if (N <= 16) return launch<io_t, 4, 4>(a, stream);
    if (N <= 32) return launch<io_t, 4, 8>(a, stream);
    if (N <= 64) return launch<io_t, 4, 16>(a, stream);
    if (N <= 128) return launch<io_t, 4, 32>(a, stream);
    return launch<io_t, 8, 32>(a, stream);
}

}  // namespace

cudaError_t launch_state_update(const StateUpdateArgs& a, bool bf16, cudaStream_t stream) {
    return bf16 ? dispatch<__nv_bfloat16>(a, stream) : dispatch<float>(a, stream);
}

}  // namespace mamba
