// Complex-state selective scan (S4D-Lin variant), sm_103a.
//
// The codechina.net overview (section 4.1) gives the complex version of the
// model the S4D-Lin initialisation A = -0.5 + i*n, and (section 5.3) keeps
// phase information in a complex state.  Per (batch b, channel d, state n):
//   A    = -exp(A_log_re[d,n]) + i * A_im[d,n]
//   h    = exp(dt * A) * h + dt * B[b,t,n] * u          (B, C complex)
//   y    = (Re(sum_n C[b,t,n] * h) + D[d] * u) * SiLU(z)
// exp(dt*A) = 2^(dt*Re A*log2 e) * (cos(dt*Im A) + i sin(dt*Im A)): one SFU
// exponential and one sine/cosine pair per state and step.  The angle
// dt*Im A reaches hundreds of radians for large steps, so its absolute error
// grows with it.  fp32 io forms the step dt and the angle in fp64 and reduces
// the angle to a quadrant there (exact to far below fp32 rounding), then takes
// sine and cosine of the fp32 remainder; bf16 io (where the output rounding is
// 2^-9) forms the angle in fp32 and reduces it to [-pi, pi] with a two-part
// 2*pi (2*pi = kTwoPiHi + kTwoPiLo in fp32).
//
// Structure (one launch): 64-thread CTAs, G lanes per chain with NPL complex
// states each, 64/G chains per CTA; the sequence runs in 16-step chunks whose
// raw inputs are loaded into registers one chunk ahead, staged to shared
// memory, and consumed by the recurrence; C.h is summed over the chain's
// lanes by a butterfly, and the element role writes y.
#include <cstdlib>

#include "common.cuh"

namespace mamba {
namespace {

constexpr int kCT = 16;     // steps per chunk
constexpr int kCNTH = 64;   // threads per CTA
constexpr float kTwoPiHi = 6.28318548202514648f;    // fp32 nearest to 2*pi
constexpr float kTwoPiLo = -1.7484556000744487e-7f; // 2*pi - kTwoPiHi
constexpr float kInvTwoPi = 0.15915494309189535f;

template <typename io_t, int NPL_, int G_>
struct CxCfg {
    static constexpr int NPL = NPL_, G = G_, T = kCT, NTH = kCNTH;
    static constexpr int CH = NTH / G;                     // chains per CTA
    static constexpr int NP = NPL * G;                     // states per chain, padded
    static constexpr int kE = T * CH;                      // elements per chunk
    static constexpr int EPT = (kE + NTH - 1) / NTH;       // consecutive steps per thread
    static constexpr int BPT = (T * NP * 2 + NTH - 1) / NTH;  // B (and C) floats per thread
    // prefetch B and C into registers only while that stays small (large
    // dstate stages them straight from global memory instead)
    static constexpr bool PREB = BPT <= 16;
    static constexpr int RB = PREB ? BPT : 1;
    // padded [t][chain] rows (EPT * kS an odd multiple of 32 / (T / EPT) mod 32)
    static constexpr int kS = ((CH + 2) / 2) % 2 == 1 ? CH + 2 : CH + 4;
    static constexpr int kF = T * kS;
    static constexpr int oDt = 0, oDu = kF, oU = 2 * kF, oYs = 3 * kF;
    // B and C as planes: [T][re | im][NP], C's imaginary plane negated
    static constexpr int oB = 4 * kF, oC = oB + T * NP * 2;
    static constexpr int kFloats = oC + T * NP * 2;
    // fp32 io only: the step dt in fp64, [t][chain] like oDt, after the floats
    static constexpr bool kDt64 = sizeof(io_t) == 4;
    static constexpr int oDt64 = (kFloats + 1) / 2;  // in doubles
    static constexpr size_t kSmem = kDt64 ? size_t(oDt64 + kF) * 8 : size_t(kFloats) * 4;
    static_assert(T % EPT == 0, "a thread's elements stay within one chain");
};

template <typename io_t>
__device__ __forceinline__ float cx_f(io_t v);
template <>
__device__ __forceinline__ float cx_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float cx_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename io_t, int NPL, int G>
struct CxRaw {
    using C = CxCfg<io_t, NPL, G>;
    io_t dl[C::EPT], u[C::EPT], z[C::EPT];
    io_t B[C::RB], Cc[C::RB];
};

struct CxArgs {
    const void *u, *delta;
    const float *A_log_re, *A_im;
    const void *B, *C;
    const float* D;
    const void* z;
    const float* delta_bias;
    void* y;
    float* last_state;
    int64_t batch, dim, seqlen;
    int dstate;
    bool softplus;
};

template <typename io_t, int NPL, int G>
__device__ __forceinline__ void cx_fetch(const CxArgs& p, CxRaw<io_t, NPL, G>& r, int b,
                                         int64_t d0, int64_t k, int tid) {
    using C = CxCfg<io_t, NPL, G>;
    const int64_t L = p.seqlen, dim = p.dim;
    const int N = p.dstate;
    const int64_t t0 = k * C::T;
    const io_t zero = io_t(0.f);
#pragma unroll
    for (int j = 0; j < C::EPT; ++j) {
        const int e = tid * C::EPT + j;
        const int c = e / C::T, t = e % C::T;
        const bool ok = e < C::kE && d0 + c < dim && t0 + t < L;
        const int64_t idx = ok ? (int64_t(b) * dim + d0 + c) * L + t0 + t : 0;
        r.dl[j] = ok ? __ldg(static_cast<const io_t*>(p.delta) + idx) : zero;
        r.u[j] = ok ? __ldg(static_cast<const io_t*>(p.u) + idx) : zero;
        r.z[j] = (ok && p.z) ? __ldg(static_cast<const io_t*>(p.z) + idx) : zero;
    }
    if constexpr (C::PREB) {
        const io_t* Bg = static_cast<const io_t*>(p.B) + int64_t(b) * L * N * 2;
        const io_t* Cg = static_cast<const io_t*>(p.C) + int64_t(b) * L * N * 2;
#pragma unroll
        for (int j = 0; j < C::BPT; ++j) {
            const int e = tid + j * C::NTH;  // [t][n][re, im] of the chunk
            const int t = e / (C::NP * 2), n = (e / 2) % C::NP, ri = e % 2;
            const bool ok = e < C::T * C::NP * 2 && n < N && t0 + t < L;
            const int64_t off = ok ? ((t0 + t) * N + n) * 2 + ri : 0;
            r.B[j] = ok ? __ldg(Bg + off) : zero;
            r.Cc[j] = ok ? __ldg(Cg + off) : zero;
        }
    }
}

// sin and cos of q * pi/2 + r to fp32 accuracy on the FMA pipe, given |r| <=
// pi/4 and the quadrant k = q mod 4: Taylor series of sin r to r^9 and of cos
// r to r^10 (next terms below 2e-10 at pi/4), then the quadrant rotates
// (sin r, cos r).
__device__ __forceinline__ void sincos_reduced(float r, int k, float& s, float& c) {
    const float r2 = r * r;
    float ps = fmaf(r2, 1.f / 362880.f, -1.f / 5040.f);
    ps = fmaf(ps, r2, 1.f / 120.f);
    ps = fmaf(ps, r2, -1.f / 6.f);
    const float sr = fmaf(ps * r2, r, r);
    float pc = fmaf(r2, -1.f / 3628800.f, 1.f / 40320.f);
    pc = fmaf(pc, r2, -1.f / 720.f);
    pc = fmaf(pc, r2, 1.f / 24.f);
    pc = fmaf(pc, r2, -0.5f);
    const float cr = fmaf(pc, r2, 1.f);
    k &= 3;
    const float a = (k & 1) ? cr : sr, b = (k & 1) ? sr : cr;
    s = (k & 2) ? -a : a;
    c = ((k + 1) & 2) ? -b : b;
}

// The angle dt * aim in fp64, written as q * pi/2 + r with |r| <= pi/4: the
// product of an fp64 step and an fp32 rate is rounded once to fp64 (2^-53
// relative), and the fp64 pi/2 (error 6e-17) keeps q * pi/2 exact to ~1e-12
// rad for any angle this scan meets, so r carries only its own fp32 rounding.
constexpr double kPio2D = 1.5707963267948966;
constexpr double kTwoOverPiD = 0.6366197723675814;
__device__ __forceinline__ void sincos_fp64_angle(double dt, float aim, float& s, float& c) {
    const double ang = dt * double(aim);
    const double q = rint(ang * kTwoOverPiD);
    const float r = float(fma(-q, kPio2D, ang));
    sincos_reduced(r, int(static_cast<long long>(q) & 3), s, c);
}

// exp(dt * (Re + i Im)) for one state: the magnitude on the SFU; the phase by
// sincos_fp64_angle (ACC: fp32 io, dt64 the step in fp64) or by the SFU's
// sine and cosine of the angle reduced to [-pi, pi] in fp32 (absolute error
// about 4e-7 per step, which a long-memory state accumulates: used for bf16
// io, where it stays far below the output's rounding)
template <bool ACC>
__device__ __forceinline__ void cx_decay(float dt, double dt64, float a2, float aim, float& ar,
                                         float& ai) {
    float s, c;
    if constexpr (ACC) {
        sincos_fp64_angle(dt64, aim, s, c);
    } else {
        const float ang = dt * aim;
        const float q = rintf(ang * kInvTwoPi);
        const float red = fmaf(-q, kTwoPiLo, fmaf(-q, kTwoPiHi, ang));
        __sincosf(red, &s, &c);
    }
    const float mag = abar_exp2<ACC>(dt * a2);
    ar = mag * c;
    ai = mag * s;
}

template <typename io_t, int NPL, int G>
__global__ void __launch_bounds__(kCNTH) scan_complex_kernel(const CxArgs p, const int dblocks) {
    using C = CxCfg<io_t, NPL, G>;
    constexpr int T = C::T, NTH = C::NTH, CH = C::CH, NP = C::NP, S = C::kS, EPT = C::EPT;
    extern __shared__ __align__(16) float sm[];
    double* smd = reinterpret_cast<double*>(sm);

    const int64_t L = p.seqlen, dim = p.dim;
    const int N = p.dstate;
    const int b = blockIdx.x / dblocks;
    const int64_t d0 = int64_t(blockIdx.x % dblocks) * CH;
    // recurrence role: chain c, states g * NPL ..; element role: chain ce, steps te0 ..
    const int tid = threadIdx.x, c = tid / G, g = tid % G;
    const int e0 = tid * EPT, ce = e0 / T, te0 = e0 % T;
    const bool e_live = e0 < C::kE && d0 + ce < dim;
    const int64_t de = e_live ? d0 + ce : 0;
    const float e_bias = (e_live && p.delta_bias) ? __ldg(p.delta_bias + de) : 0.f;
    const float e_D = (e_live && p.D) ? __ldg(p.D + de) : 0.f;
    const int64_t d = d0 + c;
    const bool chain_ok = d < dim;

    float A2[NPL], Aim[NPL], hr[NPL], hi[NPL];
    static_assert(C::kDt64 || NPL % 4 == 0, "the packed path reads B and C as float4");
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        const int n = g * NPL + i;
        const bool ok = chain_ok && n < N;
        A2[i] = ok ? -expf(__ldg(p.A_log_re + d * N + n)) * kLog2e : 0.f;
        Aim[i] = ok ? __ldg(p.A_im + d * N + n) : 0.f;
        hr[i] = hi[i] = 0.f;
    }

    // the same as pairs of states for the packed arithmetic of bf16 io
    f32x2 A2p[NPL / 2], Aim2[NPL / 2], hr2[NPL / 2], hi2[NPL / 2];
#pragma unroll
    for (int q = 0; q < NPL / 2; ++q) {
        A2p[q] = pack2(A2[2 * q], A2[2 * q + 1]);
        Aim2[q] = pack2(Aim[2 * q], Aim[2 * q + 1]);
        hr2[q] = hi2[q] = pack2(0.f, 0.f);
    }

    const int64_t nchunks = (L + T - 1) / T;
    CxRaw<io_t, NPL, G> r;
    if (nchunks > 0) cx_fetch<io_t, NPL, G>(p, r, b, d0, 0, tid);
    for (int64_t k = 0; k < nchunks; ++k) {
        const int64_t t0 = k * T;
        __syncthreads();
        float e_z[EPT];
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
            const bool ok = e_live && t0 + te0 + j < L;
            float dt;
            if constexpr (C::kDt64) {
                // fp64 step: its relative error would otherwise reach the
                // phase multiplied by the angle
                const double raw = double(cx_f(r.dl[j])) + double(e_bias);
                double dt64 = p.softplus ? (raw > 0.0 ? raw + log1p(exp(-raw)) : log1p(exp(raw)))
                                         : raw;
                if (!ok) dt64 = 0.0;
                if (e0 + j < C::kE) smd[C::oDt64 + (te0 + j) * S + ce] = dt64;
                dt = float(dt64);
            } else {
                const float raw = cx_f(r.dl[j]) + e_bias;
                dt = p.softplus ? softplus_fast(raw) : raw;
                if (!ok) dt = 0.f;
            }
            const float u = cx_f(r.u[j]);
            e_z[j] = cx_f(r.z[j]);
            if (e0 + j < C::kE) {
                sm[C::oDt + (te0 + j) * S + ce] = dt;
                sm[C::oDu + (te0 + j) * S + ce] = dt * u;
                sm[C::oU + (te0 + j) * S + ce] = u;
            }
        }
        if constexpr (C::PREB) {
#pragma unroll
            for (int j = 0; j < C::BPT; ++j) {
                const int e = tid + j * NTH;  // [t][n][re, im] of the chunk
                if (e < T * NP * 2) {
                    const int t = e / (NP * 2), n = (e / 2) % NP, ri = e % 2;
                    const int o = t * NP * 2 + ri * NP + n;
                    sm[C::oB + o] = cx_f(r.B[j]);
                    sm[C::oC + o] = ri ? -cx_f(r.Cc[j]) : cx_f(r.Cc[j]);
                }
            }
        } else {
            const io_t* Bg = static_cast<const io_t*>(p.B) + int64_t(b) * L * N * 2;
            const io_t* Cg = static_cast<const io_t*>(p.C) + int64_t(b) * L * N * 2;
            for (int e = tid; e < T * NP * 2; e += NTH) {
                const int t = e / (NP * 2), n = (e / 2) % NP, ri = e % 2;
                const bool ok = n < N && t0 + t < L;
                const int64_t off = ok ? ((t0 + t) * N + n) * 2 + ri : 0;
                const int o = t * NP * 2 + ri * NP + n;
                const float cv = ok ? Io<io_t>::load(Cg + off) : 0.f;
                sm[C::oB + o] = ok ? Io<io_t>::load(Bg + off) : 0.f;
                sm[C::oC + o] = ri ? -cv : cv;
            }
        }
        __syncthreads();
        if (k + 1 < nchunks) cx_fetch<io_t, NPL, G>(p, r, b, d0, k + 1, tid);

#pragma unroll
        for (int t = 0; t < T; ++t) {
            const float dt = sm[C::oDt + t * S + c], du = sm[C::oDu + t * S + c];
            const float* Bt = sm + C::oB + t * NP * 2 + g * NPL;  // re plane; im at + NP
            const float* Ct = sm + C::oC + t * NP * 2 + g * NPL;
            float acc = 0.f;
            if constexpr (C::kDt64) {
                const double dt64 = smd[C::oDt64 + t * S + c];
#pragma unroll
                for (int i = 0; i < NPL; ++i) {
                    float ar, ai;
                    cx_decay<true>(dt, dt64, A2[i], Aim[i], ar, ai);
                    const float nr = fmaf(ar, hr[i], fmaf(-ai, hi[i], Bt[i] * du));
                    const float ni = fmaf(ar, hi[i], fmaf(ai, hr[i], Bt[NP + i] * du));
                    hr[i] = nr;
                    hi[i] = ni;
                    acc = fmaf(Ct[i], nr, fmaf(Ct[NP + i], ni, acc));  // Ct[NP + i] = -Im C
                }
            } else {
                // pairs of states in packed f32x2 arithmetic; each state's decay
                // and update round exactly as the scalar form, and C.h sums the
                // even and the odd states separately
                const f32x2 dts = pack2(dt, dt), dus = pack2(du, du);
                f32x2 acc2 = pack2(0.f, 0.f);
#pragma unroll
                for (int v = 0; v < NPL / 4; ++v) {
                    const float4 brv = reinterpret_cast<const float4*>(Bt)[v];
                    const float4 biv = reinterpret_cast<const float4*>(Bt + NP)[v];
                    const float4 crv = reinterpret_cast<const float4*>(Ct)[v];
                    const float4 civ = reinterpret_cast<const float4*>(Ct + NP)[v];
                    const f32x2 br[2] = {pack2(brv.x, brv.y), pack2(brv.z, brv.w)};
                    const f32x2 bi[2] = {pack2(biv.x, biv.y), pack2(biv.z, biv.w)};
                    const f32x2 cr[2] = {pack2(crv.x, crv.y), pack2(crv.z, crv.w)};
                    const f32x2 ci[2] = {pack2(civ.x, civ.y), pack2(civ.z, civ.w)};
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int q = 2 * v + e;
                        // angle reduced to [-pi, pi]: ang - q 2pi with q = rint(ang / 2pi)
                        const f32x2 ang = mul2(dts, Aim2[q]);
                        float w0, w1;
                        unpack2(mul2(ang, pack2(kInvTwoPi, kInvTwoPi)), w0, w1);
                        const f32x2 qq = pack2(rintf(w0), rintf(w1));
                        float r0, r1;
                        unpack2(fma2(qq, pack2(-kTwoPiLo, -kTwoPiLo),
                                     fma2(qq, pack2(-kTwoPiHi, -kTwoPiHi), ang)),
                                r0, r1);
                        float s0, c0, s1, c1;
                        __sincosf(r0, &s0, &c0);
                        __sincosf(r1, &s1, &c1);
                        float x0, x1;
                        unpack2(mul2(dts, A2p[q]), x0, x1);
                        const f32x2 mag = pack2(ex2_approx(x0), ex2_approx(x1));
                        const f32x2 ar = mul2(mag, pack2(c0, c1)), ai = mul2(mag, pack2(s0, s1));
                        const f32x2 nai = mul2(ai, pack2(-1.f, -1.f));  // -ai, exactly
                        const f32x2 nr = fma2(ar, hr2[q], fma2(nai, hi2[q], mul2(br[e], dus)));
                        const f32x2 ni = fma2(ar, hi2[q], fma2(ai, hr2[q], mul2(bi[e], dus)));
                        hr2[q] = nr;
                        hi2[q] = ni;
                        acc2 = fma2(cr[e], nr, fma2(ci[e], ni, acc2));
                    }
                }
                float lo, hi_;
                unpack2(acc2, lo, hi_);
                acc = lo + hi_;
            }
#pragma unroll
            for (int off = G / 2; off > 0; off /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (g == 0) sm[C::oYs + t * S + c] = acc;
        }
        __syncthreads();

        // this thread's elements: y = (Re(C.h) + D u) * SiLU(z)
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
            const int t = te0 + j;
            if (!(e_live && t0 + t < L)) continue;
            const int s = t * S + ce;
            float y = fmaf(e_D, sm[C::oU + s], sm[C::oYs + s]);
            if (p.z) y = gate_silu(y, e_z[j]);
            Io<io_t>::store(static_cast<io_t*>(p.y) + (int64_t(b) * dim + de) * L + t0 + t, y);
        }
    }
    if constexpr (!C::kDt64) {
#pragma unroll
        for (int q = 0; q < NPL / 2; ++q) {
            unpack2(hr2[q], hr[2 * q], hr[2 * q + 1]);
            unpack2(hi2[q], hi[2 * q], hi[2 * q + 1]);
        }
    }
    if (chain_ok && p.last_state) {
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            const int n = g * NPL + i;
            if (n < N)
                *reinterpret_cast<float2*>(p.last_state + ((int64_t(b) * dim + d) * N + n) * 2) =
                    make_float2(hr[i], hi[i]);
        }
    }
}

template <typename io_t, int NPL, int G>
cudaError_t launch_cx(const CxArgs& p, cudaStream_t stream) {
    using C = CxCfg<io_t, NPL, G>;
    const int64_t dblocks = (p.dim + C::CH - 1) / C::CH;
    const int64_t blocks = dblocks * p.batch;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    cudaError_t err = cudaFuncSetAttribute(scan_complex_kernel<io_t, NPL, G>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           int(C::kSmem));
    if (err != cudaSuccess) return err;
    scan_complex_kernel<io_t, NPL, G><<<unsigned(blocks), C::NTH, C::kSmem, stream>>>(p, int(dblocks));
    return cudaGetLastError();
}

// Tile by dstate.  At dstate 16 the fp32 path (sine and cosine on the FMA
// pipe, ~20 instructions per state and step) runs faster with 2 states x 8
// lanes (more warps to hide its latency: 975 vs 1220 us on the 130M-style
// shape); the bf16 path (SFU sine/cosine) with 4 x 4 (604 vs 738 us).
template <typename io_t>
cudaError_t dispatch_cx(const CxArgs& p, cudaStream_t stream) {
    const int N = p.dstate;
    if (N <= 8) return launch_cx<io_t, 4, 2>(p, stream);
    if (N <= 16) {
        if constexpr (sizeof(io_t) == 4) return launch_cx<io_t, 2, 8>(p, stream);
        return launch_cx<io_t, 4, 4>(p, stream);
    }
    if (N <= 32) return launch_cx<io_t, 4, 8>(p, stream);
    if (N <= 64) return launch_cx<io_t, 4, 16>(p, stream);
    if (N <= 128) return launch_cx<io_t, 4, 32>(p, stream);
    return launch_cx<io_t, 8, 32>(p, stream);
}

}  // namespace

cudaError_t launch_scan_complex(const void* u, const void* delta, const float* A_log_re,
                                const float* A_im, const void* B, const void* C, const float* D,
                                const void* z, const float* delta_bias, bool softplus, void* y,
                                float* last_state, int64_t batch, int64_t dim, int64_t seqlen,
                                int dstate, bool bf16, cudaStream_t stream) {
    const CxArgs p{u, delta, A_log_re, A_im, B, C, D, z, delta_bias, y, last_state,
                   batch, dim, seqlen, dstate, softplus};
    return bf16 ? dispatch_cx<__nv_bfloat16>(p, stream) : dispatch_cx<float>(p, stream);
}

}  // namespace mamba
