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

template <typename io_t, int NPL, int G, bool VEC>
__global__ void __launch_bounds__(256) state_update_kernel(StateUpdateArgs p) {
    const int64_t chains = p.batch * p.dim;
    const int64_t gtid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t chain = gtid / G;
    const int g = int(gtid % G);
    // Whole G-lane groups are inside or outside together (G divides 32 and the
    // block size), so the shuffles below never mix live and dead lanes.
    if (chain >= chains) return;
    const int64_t b = chain / p.dim, d = chain % p.dim;
    const int N = p.dstate;

    const float raw = Io<io_t>::load(static_cast<const io_t*>(p.dt) + chain) +
                      (p.dt_bias ? __ldg(p.dt_bias + d) : 0.f);
    const float dt = !p.softplus ? raw : sizeof(io_t) == 2 ? softplus_fast(raw) : softplus_accurate(raw);
    const float x = Io<io_t>::load(static_cast<const io_t*>(p.x) + chain);
    const float dx = dt * x;
    const io_t* Bb = static_cast<const io_t*>(p.B) + b * N;
    const io_t* Cb = static_cast<const io_t*>(p.C) + b * N;
    float* st = p.state + chain * N + g * NPL;

    float h[NPL];
    if constexpr (VEC) {
#pragma unroll
        for (int i = 0; i < NPL; i += 4) {
            const float4 v = *reinterpret_cast<const float4*>(st + i);
            h[i] = v.x; h[i + 1] = v.y; h[i + 2] = v.z; h[i + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < NPL; ++i) h[i] = (g * NPL + i < N) ? st[i] : 0.f;
    }

    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        const int n = g * NPL + i;
        if (VEC || n < N) {
            // A = -exp(A_log) = -2^(A_log * log2 e); Abar = 2^(dt * A * log2 e)
            const float A2 = -ex2_approx(__ldg(p.A_log + d * N + n) * kLog2e) * kLog2e;
            const float a = ex2_approx(dt * A2);
            h[i] = fmaf(a, h[i], dx * Io<io_t>::load(Bb + n));
            acc = fmaf(Io<io_t>::load(Cb + n), h[i], acc);
        }
    }

    if constexpr (VEC) {
#pragma unroll
        for (int i = 0; i < NPL; i += 4)
            *reinterpret_cast<float4*>(st + i) = make_float4(h[i], h[i + 1], h[i + 2], h[i + 3]);
    } else {
#pragma unroll
        for (int i = 0; i < NPL; ++i)
            if (g * NPL + i < N) st[i] = h[i];
    }

    // Lanes of this chain's group (all live together, see above).
    const unsigned lane = threadIdx.x & 31u;
    const unsigned gmask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (lane / G * G));
#pragma unroll
    for (int off = G / 2; off > 0; off /= 2) acc += __shfl_xor_sync(gmask, acc, off, G);

    if (g == 0) {
        if (p.D) acc = fmaf(__ldg(p.D + d), x, acc);
        if (p.z) acc *= silu_fast(Io<io_t>::load(static_cast<const io_t*>(p.z) + chain));
        Io<io_t>::store(static_cast<io_t*>(p.out) + chain, acc);
    }
}

template <typename io_t, int NPL, int G>
cudaError_t launch(const StateUpdateArgs& a, cudaStream_t stream) {
    const int64_t threads = a.batch * a.dim * G;
    const int64_t blocks = (threads + 255) / 256;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const bool vec = (a.dstate % 4 == 0) && (a.dstate == NPL * G) &&
                     (reinterpret_cast<uintptr_t>(a.state) % 16 == 0);
    if (vec)
        state_update_kernel<io_t, NPL, G, true><<<unsigned(blocks), 256, 0, stream>>>(a);
    else
        state_update_kernel<io_t, NPL, G, false><<<unsigned(blocks), 256, 0, stream>>>(a);
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
