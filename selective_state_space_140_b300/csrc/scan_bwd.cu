// Backward of the selective scan (training), sm_103a.
//
// The codechina.net overview (section 2.2, point 3) trains the scan by not
// keeping the forward's intermediate states and recomputing them in the
// backward pass.  One kernel does both halves for a group of chains:
//
//   forward phase  -- the recurrence over the whole sequence, storing only the
//                     state at the start of every 16-step chunk (a checkpoint,
//                     N floats per chain per chunk, in scratch memory);
//   reverse phase  -- for chunk k = last .. 0: recompute the chunk's 16 states
//                     from its checkpoint into shared memory, then run the
//                     adjoint recurrence backwards through the chunk
//                       g_tn = dy_t C_tn + Abar_{t+1,n} g_{t+1,n}
//                     and form every gradient of the step (see the fp64
//                     oracle, which writes the same chain rule out).
//
// B, C, A_log, D and the bias are shared by many chains, so their gradients
// are sums: dB and dC over the channels of a batch row are reduced across the
// warp's chains with shuffles (a halving "transpose" reduction that leaves one
// sum per lane) and across the CTA's warps in shared memory, then added to the
// fp32 outputs with one global atomic per value and chunk; dA_log, dD and the
// bias gradient accumulate in registers over the whole sequence and are added
// once at the end.
#include <cstdlib>

#include "common.cuh"

namespace mamba {
namespace {

constexpr int kBT = 16;     // steps per chunk
constexpr int kBNTH = 64;   // threads per CTA

template <typename io_t, int NPL_, int G_>
struct BwdCfg {
    static constexpr int NPL = NPL_, G = G_, T = kBT, NTH = kBNTH;
    static constexpr int CH = NTH / G;        // chains per CTA
    static constexpr int CPW = 32 / G;        // chains per warp
    static constexpr int NW = NTH / 32;       // warps
    static constexpr int NP = NPL * G;        // states per chain, padded
    static constexpr int NQ = NPL / 4;        // float4 per thread per step
    // shared memory (floats)
    static constexpr int kE = T * CH;                 // one per-element field
    static constexpr int oDt = 0, oDu = kE, oU = 2 * kE, oDy = 3 * kE, oDout = 4 * kE;
    static constexpr int oSilu = 5 * kE, oDsilu = 6 * kE, oSp = 7 * kE;
    static constexpr int oGu = 8 * kE, oGdt = 9 * kE;  // reduced sum_n g B, sum_n g (...)
    static constexpr int oB = 10 * kE, oC = oB + T * NP;
    static constexpr int oH = oC + T * NP;              // [T][NQ][NTH] float4 states
    static constexpr int oYs = oH + T * NQ * NTH * 4;  // [T][NTH] partial C.h
    static constexpr int oRed = oYs + T * NTH;         // [NW][T][2][NP] per-warp dB/dC sums
    static constexpr int kFloats = oRed + NW * T * 2 * NP;
    static constexpr size_t kSmem = size_t(kFloats) * 4;
    static_assert(NPL % 4 == 0, "states per lane in whole float4");
};

struct BwdArgs : ScanBwdArgs {
    float* ckpt;  // [batch * dim][nchunks][N] scratch: state at each chunk start
};

// Per-element inputs of chunk k into shared memory: dt (and, for the reverse
// phase, u, dout and the gate values).  Chains past dim and steps past L get
// dt = 0, u = 0, dout = 0, so they leave every gradient untouched.
template <typename io_t, int NPL, int G, bool REVERSE>
__device__ __forceinline__ void load_chunk(const BwdArgs& a, float* sm, int b, int64_t d0,
                                           int64_t k, int tid) {
    using C = BwdCfg<io_t, NPL, G>;
    const ScanArgs& p = a.f;
    const int64_t L = p.seqlen, dim = p.dim;
    const int N = p.dstate;
    const int64_t t0 = k * C::T;
    for (int e = tid; e < C::kE; e += C::NTH) {
        const int c = e / C::T, t = e % C::T;   // consecutive threads walk time
        const int64_t d = d0 + c;
        const bool ok = d < dim && t0 + t < L;
        const int64_t idx = (int64_t(b) * dim + (ok ? d : 0)) * L + (ok ? t0 + t : 0);
        float dt = 0.f, u = 0.f, sp = 0.f;
        if (ok) {
            const float raw = Io<io_t>::load(static_cast<const io_t*>(p.delta) + idx) +
                              (p.delta_bias ? __ldg(p.delta_bias + d) : 0.f);
            dt = p.softplus ? (sizeof(io_t) == 2 ? softplus_fast(raw) : softplus_accurate(raw))
                            : raw;
            sp = p.softplus ? rcp_approx(1.f + ex2_approx(-raw * kLog2e)) : 1.f;  // softplus'
            u = Io<io_t>::load(static_cast<const io_t*>(p.u) + idx);
        }
        const int s = t * C::CH + c;  // [t][c]
        sm[C::oDt + s] = dt;
        sm[C::oDu + s] = dt * u;
        if constexpr (REVERSE) {
            sm[C::oU + s] = u;
            sm[C::oSp + s] = sp;
            const float go = ok ? Io<io_t>::load(static_cast<const io_t*>(a.dout) + idx) : 0.f;
            sm[C::oDout + s] = go;
            float silu = 1.f, dsilu = 0.f;
            if (p.z && ok) {
                const float z = Io<io_t>::load(static_cast<const io_t*>(p.z) + idx);
                const float sg = rcp_approx(1.f + ex2_approx(-z * kLog2e));
                silu = z * sg;
                dsilu = sg * (1.f + z * (1.f - sg));
            }
            sm[C::oSilu + s] = silu;
            sm[C::oDsilu + s] = dsilu;
        }
    }
    // B (and C) of the chunk, fp32 [t][n], zero past L and past N
    const io_t* Bg = static_cast<const io_t*>(p.B) + int64_t(b) * L * N;
    const io_t* Cg = static_cast<const io_t*>(p.C) + int64_t(b) * L * N;
    for (int e = tid; e < C::T * C::NP; e += C::NTH) {
        const int t = e / C::NP, n = e % C::NP;
        const bool ok = n < N && t0 + t < L;
        sm[C::oB + e] = ok ? Io<io_t>::load(Bg + (t0 + t) * N + n) : 0.f;
        if constexpr (REVERSE) sm[C::oC + e] = ok ? Io<io_t>::load(Cg + (t0 + t) * N + n) : 0.f;
    }
}

// Sum of V values per lane over the CPW chains of a warp (lane = chain * G +
// g; lanes with the same g hold the same value indices).  Each round halves
// the values a lane keeps: the lanes whose chain bit M is set keep the upper
// half and send the lower half to the partner chain (chain ^ M), which does
// the opposite, and both add what they receive.  When one value is left, the
// remaining rounds are a plain butterfly.  At the end the lane of chain cw
// holds the sums of value indices [cw * V / CPW, (cw + 1) * V / CPW) when
// V >= CPW, else the sum of index cw / (CPW / V) (shared by CPW / V lanes).
template <int V, int M, int G>
struct ChainSum {
    static __device__ __forceinline__ void run(float* v, int cw) {
        if constexpr (M >= 1) {
            if constexpr (V > 1) {
                constexpr int H = V / 2;
                const bool up = (cw & M) != 0;
#pragma unroll
                for (int i = 0; i < H; ++i) {
                    const float send = up ? v[i] : v[i + H];
                    const float keep = up ? v[i + H] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, M * G);
                }
                ChainSum<H, M / 2, G>::run(v, cw);
            } else {
                v[0] += __shfl_xor_sync(0xffffffffu, v[0], M * G);
                ChainSum<1, M / 2, G>::run(v, cw);
            }
        }
    }
};

template <typename io_t, int NPL, int G>
__global__ void __launch_bounds__(kBNTH) scan_bwd_kernel(const BwdArgs a, const int dblocks) {
    using C = BwdCfg<io_t, NPL, G>;
    constexpr int T = C::T, NTH = C::NTH, CH = C::CH, NP = C::NP, NQ = C::NQ, CPW = C::CPW;
    constexpr int V = 2 * NPL;  // dB and dC values per lane and step
    extern __shared__ __align__(16) float sm[];
    float* sDacc = sm + C::kFloats;       // [CH] per-chain sum of dy * u
    float* sBacc = sDacc + CH;            // [CH] per-chain sum of ddelta
    float4* sH = reinterpret_cast<float4*>(sm + C::oH);

    const ScanArgs& p = a.f;
    const int64_t L = p.seqlen, dim = p.dim;
    const int N = p.dstate;
    const int b = blockIdx.x / dblocks;
    const int64_t d0 = int64_t(blockIdx.x % dblocks) * CH;
    const int tid = threadIdx.x, c = tid / G, g = tid % G;
    const int warp = tid / 32, cw = (tid % 32) / G;
    const int64_t d = d0 + c;
    const bool chain_ok = d < dim;
    const int64_t chain = int64_t(b) * dim + (chain_ok ? d : 0);
    const int64_t nchunks = (L + T - 1) / T;
    float* ck = a.ckpt + chain * nchunks * N;

    float A[NPL], A2[NPL], h[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        const int n = g * NPL + i;
        A[i] = (chain_ok && n < N) ? -expf(__ldg(p.A_log + d * N + n)) : 0.f;
        A2[i] = A[i] * kLog2e;
        h[i] = 0.f;
    }
    for (int e = tid; e < 2 * CH; e += NTH) sDacc[e] = 0.f;

    // ---------------- forward phase: checkpoints ----------------
    for (int64_t k = 0; k < nchunks; ++k) {
        __syncthreads();
        load_chunk<io_t, NPL, G, false>(a, sm, b, d0, k, tid);
        __syncthreads();
        if (chain_ok) {
#pragma unroll
            for (int i = 0; i < NPL; ++i)
                if (g * NPL + i < N) ck[k * N + g * NPL + i] = h[i];
        }
        const int tlen = L - k * T < T ? int(L - k * T) : T;
        for (int t = 0; t < tlen; ++t) {
            const float dt = sm[C::oDt + t * CH + c], du = sm[C::oDu + t * CH + c];
#pragma unroll
            for (int i = 0; i < NPL; ++i)
                h[i] = fmaf(ex2_approx(dt * A2[i]), h[i], du * sm[C::oB + t * NP + g * NPL + i]);
        }
    }

    // ---------------- reverse phase ----------------
    float gc[NPL], dA[NPL];  // Abar_{t+1} g_{t+1}; sum of g dt Abar h_{t-1}
#pragma unroll
    for (int i = 0; i < NPL; ++i) gc[i] = dA[i] = 0.f;
    for (int64_t k = nchunks - 1; k >= 0; --k) {
        __syncthreads();
        load_chunk<io_t, NPL, G, true>(a, sm, b, d0, k, tid);
        float hs[NPL];  // state at the start of the chunk
#pragma unroll
        for (int i = 0; i < NPL; ++i)
            hs[i] = (chain_ok && g * NPL + i < N) ? ck[k * N + g * NPL + i] : 0.f;
        __syncthreads();
        const int tlen = L - k * T < T ? int(L - k * T) : T;
        const int64_t t0 = k * T;

        // recompute the chunk's states (kept in shared memory) and C.h partials
        {
            float hh[NPL];
#pragma unroll
            for (int i = 0; i < NPL; ++i) hh[i] = hs[i];
            for (int t = 0; t < tlen; ++t) {
                const float dt = sm[C::oDt + t * CH + c], du = sm[C::oDu + t * CH + c];
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < NPL; ++i) {
                    const int n = g * NPL + i;
                    hh[i] = fmaf(ex2_approx(dt * A2[i]), hh[i], du * sm[C::oB + t * NP + n]);
                    acc = fmaf(sm[C::oC + t * NP + n], hh[i], acc);
                }
#pragma unroll
                for (int q = 0; q < NQ; ++q)
                    sH[(t * NQ + q) * NTH + tid] =
                        make_float4(hh[4 * q], hh[4 * q + 1], hh[4 * q + 2], hh[4 * q + 3]);
                sm[C::oYs + t * NTH + tid] = acc;
            }
        }
        __syncthreads();

        // per element: y = C.h + D u, the gate's gradient, dy
        for (int e = tid; e < C::kE; e += NTH) {
            const int ce = e / T, t = e % T;
            const int64_t de = d0 + ce;
            if (t >= tlen) continue;
            const int s = t * CH + ce;
            float ys = 0.f;
#pragma unroll
            for (int gg = 0; gg < G; ++gg) ys += sm[C::oYs + t * NTH + ce * G + gg];
            const float u = sm[C::oU + s], go = sm[C::oDout + s];
            const float y = p.D && de < dim ? fmaf(__ldg(p.D + de), u, ys) : ys;
            if (p.z) {
                if (de < dim)
                    Io<io_t>::store(static_cast<io_t*>(a.dz) + (int64_t(b) * dim + de) * L + t0 + t,
                                    go * y * sm[C::oDsilu + s]);
                sm[C::oDy + s] = go * sm[C::oSilu + s];
            } else {
                sm[C::oDy + s] = go;
            }
        }
        __syncthreads();

        // adjoint, backwards through the chunk
        for (int t = tlen - 1; t >= 0; --t) {
            const int s = t * CH + c;
            const float dy = sm[C::oDy + s], dt = sm[C::oDt + s], u = sm[C::oU + s];
            const float dtu = dt * u;
            float hp[NPL], hc[NPL];
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const float4 vc = sH[(t * NQ + q) * NTH + tid];
                hc[4 * q] = vc.x; hc[4 * q + 1] = vc.y; hc[4 * q + 2] = vc.z; hc[4 * q + 3] = vc.w;
                if (t > 0) {
                    const float4 vp = sH[((t - 1) * NQ + q) * NTH + tid];
                    hp[4 * q] = vp.x; hp[4 * q + 1] = vp.y; hp[4 * q + 2] = vp.z; hp[4 * q + 3] = vp.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) hp[4 * q + e] = hs[4 * q + e];
                }
            }
            float v[V];
            float gu = 0.f, gd = 0.f;
#pragma unroll
            for (int i = 0; i < NPL; ++i) {
                const int n = g * NPL + i;
                const float Bn = sm[C::oB + t * NP + n], Cn = sm[C::oC + t * NP + n];
                const float ab = ex2_approx(dt * A2[i]);
                const float gn = fmaf(dy, Cn, gc[i]);
                const float ahp = ab * hp[i];
                v[i] = gn * dtu;        // dB
                v[NPL + i] = dy * hc[i];  // dC
                gu = fmaf(gn, Bn, gu);
                gd = fmaf(gn, fmaf(A[i], ahp, u * Bn), gd);
                dA[i] = fmaf(gn * dt, ahp, dA[i]);
                gc[i] = ab * gn;
            }
#pragma unroll
            for (int off = G / 2; off > 0; off /= 2) {
                gu += __shfl_xor_sync(0xffffffffu, gu, off);
                gd += __shfl_xor_sync(0xffffffffu, gd, off);
            }
            if (g == 0) {
                sm[C::oGu + s] = gu;
                sm[C::oGdt + s] = gd;
            }
            ChainSum<V, CPW / 2, G>::run(v, cw);
            float* red = sm + C::oRed + (warp * T + t) * 2 * NP;  // [q][n]
            if constexpr (V >= CPW) {
                constexpr int K = V / CPW;
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    const int idx = cw * K + j, q = idx / NPL, n = g * NPL + idx % NPL;
                    red[q * NP + n] = v[j];
                }
            } else {
                constexpr int R = CPW / V;
                if (cw % R == 0) {
                    const int idx = cw / R, q = idx / NPL, n = g * NPL + idx % NPL;
                    red[q * NP + n] = v[0];
                }
            }
        }
        __syncthreads();

        // per element: du, ddelta; per chain: sums for dD and the bias gradient
        for (int e = tid; e < C::kE; e += NTH) {
            const int ce = e / T, t = e % T;
            const int64_t de = d0 + ce;
            if (t >= tlen || de >= dim) continue;
            const int s = t * CH + ce;
            const int64_t idx = (int64_t(b) * dim + de) * L + t0 + t;
            const float dy = sm[C::oDy + s], u = sm[C::oU + s];
            const float du = fmaf(sm[C::oDt + s], sm[C::oGu + s],
                                  p.D ? dy * __ldg(p.D + de) : 0.f);
            const float dr = sm[C::oGdt + s] * sm[C::oSp + s];
            Io<io_t>::store(static_cast<io_t*>(a.du) + idx, du);
            Io<io_t>::store(static_cast<io_t*>(a.ddelta) + idx, dr);
            atomicAdd(&sDacc[ce], dy * u);
            atomicAdd(&sBacc[ce], dr);
        }
        // dB, dC of the chunk: sum over the warps, then one atomic per value
        for (int e = tid; e < T * 2 * NP; e += NTH) {
            const int t = e / (2 * NP), q = (e / NP) % 2, n = e % NP;
            if (t >= tlen || n >= N) continue;
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < C::NW; ++w) sum += sm[C::oRed + (w * T + t) * 2 * NP + q * NP + n];
            atomicAdd((q ? a.dC : a.dB) + (int64_t(b) * L + t0 + t) * N + n, sum);
        }
    }

    // dA_log = dA * A (A = -exp(A_log)); dD, the bias gradient: per chain sums
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        const int n = g * NPL + i;
        if (chain_ok && n < N) atomicAdd(a.dA_log + d * N + n, dA[i] * A[i]);
    }
    __syncthreads();
    if (g == 0 && chain_ok) {
        if (a.dD) atomicAdd(a.dD + d, sDacc[c]);
        if (a.ddelta_bias) atomicAdd(a.ddelta_bias + d, sBacc[c]);
    }
}

template <typename io_t, int NPL, int G>
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream) {
    using C = BwdCfg<io_t, NPL, G>;
    const int64_t dblocks = (a.f.dim + C::CH - 1) / C::CH;
    const int64_t blocks = dblocks * a.f.batch;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const size_t smem = C::kSmem + 2 * C::CH * sizeof(float);
    cudaError_t err = cudaFuncSetAttribute(scan_bwd_kernel<io_t, NPL, G>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (err != cudaSuccess) return err;
    scan_bwd_kernel<io_t, NPL, G><<<unsigned(blocks), C::NTH, smem, stream>>>(a, int(dblocks));
    return cudaGetLastError();
}

template <typename io_t>
cudaError_t dispatch_bwd(const BwdArgs& a, cudaStream_t stream) {
    const int N = a.f.dstate;
    if (N <= 8) return launch_bwd<io_t, 4, 2>(a, stream);
    if (N <= 16) return launch_bwd<io_t, 8, 2>(a, stream);
    if (N <= 32) return launch_bwd<io_t, 8, 4>(a, stream);
    if (N <= 64) return launch_bwd<io_t, 8, 8>(a, stream);
    if (N <= 128) return launch_bwd<io_t, 8, 16>(a, stream);
    return launch_bwd<io_t, 8, 32>(a, stream);
}

}  // namespace

cudaError_t launch_scan_bwd(const ScanBwdArgs& s, bool bf16, cudaStream_t stream) {
    const int64_t chains = s.f.batch * s.f.dim;
    const int64_t nchunks = (s.f.seqlen + kBT - 1) / kBT;
    cudaError_t err = cudaSuccess;
    // the shared-parameter gradients are sums: start them at zero
    const size_t nbc = size_t(s.f.batch) * s.f.seqlen * s.f.dstate * sizeof(float);
    if (nbc && (err = cudaMemsetAsync(s.dB, 0, nbc, stream)) != cudaSuccess) return err;
    if (nbc && (err = cudaMemsetAsync(s.dC, 0, nbc, stream)) != cudaSuccess) return err;
    if (s.f.dim &&
        (err = cudaMemsetAsync(s.dA_log, 0, size_t(s.f.dim) * s.f.dstate * 4, stream)) != cudaSuccess)
        return err;
    if (s.dD && s.f.dim && (err = cudaMemsetAsync(s.dD, 0, size_t(s.f.dim) * 4, stream)) != cudaSuccess)
        return err;
    if (s.ddelta_bias && s.f.dim &&
        (err = cudaMemsetAsync(s.ddelta_bias, 0, size_t(s.f.dim) * 4, stream)) != cudaSuccess)
        return err;
    if (chains == 0 || nchunks == 0) return cudaSuccess;
    // checkpoints: the state at the start of every chunk, stream-ordered scratch
    void* ck = nullptr;
    const size_t ckb = size_t(chains) * nchunks * s.f.dstate * sizeof(float);
    if ((err = cudaMallocAsync(&ck, ckb, stream)) != cudaSuccess) return err;
    BwdArgs a;
    static_cast<ScanBwdArgs&>(a) = s;
    a.ckpt = static_cast<float*>(ck);
    err = bf16 ? dispatch_bwd<__nv_bfloat16>(a, stream) : dispatch_bwd<float>(a, stream);
    const cudaError_t ferr = cudaFreeAsync(ck, stream);
    return err != cudaSuccess ? err : ferr;
}

}  // namespace mamba
