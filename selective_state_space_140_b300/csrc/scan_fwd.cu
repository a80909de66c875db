// Fused selective-scan forward kernel for sm_103a.
//
// One launch does every step of the scan: dt = softplus(delta + bias),
// Abar = exp(dt*A) with A = -exp(A_log), Bbar u = dt*B*u, the recurrence
// h = Abar h + Bbar u, y = C.h + D u, the SiLU(z) gate and the final state
// (codechina.net overview, section 1 "硬件感知算法" and section 2.2 "核融合":
// parameters are read from HBM once, discretisation and recurrence happen on
// chip, and only the result is written).  Only u, delta, z, B, C are read and
// only y and the last state are written.
//
// Work decomposition.  Every (batch, channel) chain is an independent
// recurrence over `dstate` independent states.  A thread owns NPL states of
// one chain and walks the whole sequence in order, so the fp32 state never
// leaves registers and no inter-thread scan is needed (the sequential
// recurrence of the pages, with the parallelism taken across batch, channel
// and state instead of across time).  G threads share a chain, CH chains
// share a CTA, and the chains of a CTA belong to one batch so that one copy
// of B and C in shared memory serves all of them.
//
// The sequence is processed in chunks of T steps; per chunk:
//   A. B and C of the chunk have been brought into shared memory by a bulk
//      copy (TMA, cp.async.bulk) issued two chunks ahead; bf16 values are
//      widened once to fp32.  Each thread turns its 128-bit register-prefetched
//      slice of delta and u into (dt, dt*u) for all states and issues the
//      128-bit loads of the next chunk's delta, u, z.
//   B. The recurrence, two states per packed f32x2 instruction: per step and
//      state one ex2 on the SFU, a multiply for dt*A, a multiply for dt*u*B,
//      an fma for h and an fma for the C contraction.  Each thread leaves one
//      partial sum of C.h per step in shared memory.
//   C. Per (chain, step): sum the G partials, add D*u, gate with SiLU(z),
//      round and store y with 128-bit stores.
#include <type_traits>

#include "common.cuh"

namespace mamba {

// Error word of this kernel family (see mbar_wait).
__device__ unsigned int g_scan_error;

namespace {

template <typename io_t, int NPL_, int G_, int CH_, int T_>
struct Cfg {
    using io = io_t;
    static constexpr int NPL = NPL_, G = G_, CH = CH_, T = T_;
    static constexpr int NTH = CH * G;
    static constexpr int NP = NPL * G;          // padded states per chain
    static constexpr int VEC = Io<io_t>::kVec;  // io elements per 16 bytes
    static constexpr int SEGROW = T / VEC;      // 16-byte segments per chain per chunk
    static constexpr int NSEG = CH * SEGROW;
    static constexpr int SPT = (NSEG + NTH - 1) / NTH;
    static constexpr int ES = sizeof(io_t);
    static constexpr int NQ = NPL / 4;          // quads of states per thread
    static_assert(NPL % 4 == 0 && T % VEC == 0 && T % 4 == 0, "tile shape");
    static_assert((T / 4 & (T / 4 - 1)) == 0, "T/4 must be a power of two");
    // shared memory layout (bytes)
    static constexpr size_t kBar = 0;                                   // 2 mbarriers
    static constexpr size_t kStage = 128;                               // 2 x (B, C) raw
    static constexpr size_t kStageBytes = size_t(T) * NP * ES;         // one array, one chunk
    static constexpr size_t kBf = kStage + 4 * kStageBytes;             // fp32 B, C
    static constexpr size_t kBfBytes = size_t(T) * NP * 4;
    static constexpr size_t kDu = kBf + 2 * kBfBytes;                   // (dt,dt,du,du)
    static constexpr size_t kY = kDu + size_t(T) * CH * 16;             // partial sums
    static constexpr size_t kSmem = kY + size_t(NTH) * T * 4;
    // DIRECT configurations (fp32 io with dstate == NP) skip the fp32 copy
    static constexpr size_t kSmemDirect = kDu - 2 * kBfBytes + size_t(T) * CH * 16 +
                                          size_t(NTH) * T * 4;
};

// Swizzle of the 16-byte chunk index within a row of partial sums, so that
// both the per-step writes (consecutive rows) and the per-chain reads (rows
// G apart) of one warp land in distinct banks.
template <int T>
__device__ __forceinline__ int yswz(int row) {
    return (row ^ (row >> 2)) & (T / 4 - 1);
}

struct Layout {
    uint64_t* bar;
    unsigned char* stage;  // [2][B|C] raw io values, [T][N]
    float* bf;             // [2 arrays][T][NP] fp32 (or the stage itself when DIRECT)
    float4* du;            // [T][CH]
    float* y;              // [NTH][T] swizzled
};

// 128-bit (or element-wise, at ragged edges) load of VEC consecutive io values.
template <typename C, bool VECIO>
__device__ __forceinline__ uint4 load_seg(const typename C::io* row, int64_t t, int64_t L,
                                          bool valid) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (!valid) return v;
    if (VECIO) {
        if (t + C::VEC <= L) v = __ldg(reinterpret_cast<const uint4*>(row + t));
        return v;
    }
    unsigned w[4] = {0u, 0u, 0u, 0u};
    if constexpr (C::ES == 4) {
        const unsigned* r = reinterpret_cast<const unsigned*>(row);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (t + e < L) w[e] = __ldg(r + t + e);
    } else {
        const unsigned short* r = reinterpret_cast<const unsigned short*>(row);
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (t + e < L) w[e >> 1] |= unsigned(__ldg(r + t + e)) << (16 * (e & 1));
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename C, bool VECIO>
__device__ __forceinline__ void store_seg(typename C::io* row, int64_t t, int64_t L,
                                          const float (&val)[C::VEC]) {
    if constexpr (C::ES == 4) {
        if (VECIO && t + 4 <= L) {
            *reinterpret_cast<float4*>(row + t) = make_float4(val[0], val[1], val[2], val[3]);
            return;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (t + e < L) reinterpret_cast<float*>(row)[t + e] = val[e];
    } else {
        unsigned w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const __nv_bfloat162 p = __floats2bfloat162_rn(val[2 * q], val[2 * q + 1]);
            w[q] = *reinterpret_cast<const unsigned*>(&p);
        }
        if (VECIO && t + 8 <= L) {
            *reinterpret_cast<uint4*>(row + t) = make_uint4(w[0], w[1], w[2], w[3]);
            return;
        }
        unsigned short* r = reinterpret_cast<unsigned short*>(row);
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (t + e < L) r[t + e] = static_cast<unsigned short>(w[e >> 1] >> (16 * (e & 1)));
    }
}

template <typename io_t, int NPL, int G, int CH, int T, bool VECIO, bool DIRECT>
__global__ void __launch_bounds__(CH* G)
    scan_fwd_kernel(const ScanArgs p, const int dblocks, const int tma_ok) {
    using C = Cfg<io_t, NPL, G, CH, T>;
    constexpr int NTH = C::NTH, NP = C::NP, VEC = C::VEC, NQ = C::NQ;
    extern __shared__ __align__(128) unsigned char smem[];
    Layout s;
    s.bar = reinterpret_cast<uint64_t*>(smem + C::kBar);
    s.stage = smem + C::kStage;
    s.bf = reinterpret_cast<float*>(smem + C::kBf);
    s.du = reinterpret_cast<float4*>(smem + (DIRECT ? C::kBf : C::kDu));
    s.y = reinterpret_cast<float*>(smem + (DIRECT ? C::kBf + size_t(T) * CH * 16 : C::kY));

    const int64_t L = p.seqlen, dim = p.dim;
    const int N = p.dstate;
    const int b = blockIdx.x / dblocks;
    const int64_t d0 = int64_t(blockIdx.x % dblocks) * CH;
    const int tid = threadIdx.x;
    const int c = tid / G, g = tid % G;
    const int64_t d = d0 + c;
    const bool chain_ok = d < dim;
    const int64_t nchunks = (L + T - 1) / T;

    const io_t* Bg = static_cast<const io_t*>(p.B) + int64_t(b) * L * N;
    const io_t* Cg = static_cast<const io_t*>(p.C) + int64_t(b) * L * N;
    const uint32_t stage_bytes = uint32_t(T) * N * C::ES;

    auto stageB = [&](int k) { return s.stage + size_t(2 * (k & 1)) * C::kStageBytes; };
    auto stageC = [&](int k) { return s.stage + size_t(2 * (k & 1) + 1) * C::kStageBytes; };
    auto chunk_by_tma = [&](int64_t k) { return tma_ok && (k + 1) * T <= L; };
    auto issue = [&](int64_t k) {  // thread 0 only
        const int64_t off = k * T * N;
        mbar_arrive_expect_tx(&s.bar[k & 1], 2 * stage_bytes);
        bulk_g2s(stageB(int(k)), Bg + off, stage_bytes, &s.bar[k & 1]);
        bulk_g2s(stageC(int(k)), Cg + off, stage_bytes, &s.bar[k & 1]);
    };

    if (tid == 0) {
        mbar_init(&s.bar[0], 1);
        mbar_init(&s.bar[1], 1);
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncthreads();
    if (tid == 0) {
        if (nchunks > 0 && chunk_by_tma(0)) issue(0);
        if (nchunks > 1 && chunk_by_tma(1)) issue(1);
    }

    // Per-thread constants: A2 = -exp(A_log) * log2(e), so Abar = 2^(dt*A2).
    f32x2 A2[2 * NQ], h[2 * NQ];
#pragma unroll
    for (int q = 0; q < 2 * NQ; ++q) {
        float a[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int n = g * NPL + 2 * q + e;
            a[e] = (chain_ok && n < N) ? -expf(__ldg(p.A_log + d * N + n)) * kLog2e : 0.f;
        }
        A2[q] = pack2(a[0], a[1]);
        h[q] = pack2(0.f, 0.f);
    }

    // Register prefetch of delta, u, z: slice s = tid + i*NTH is chain
    // s % CH, 16-byte segment s / CH of the chunk.
    const io_t* dl = static_cast<const io_t*>(p.delta);
    const io_t* uu = static_cast<const io_t*>(p.u);
    const io_t* zz = static_cast<const io_t*>(p.z);
    io_t* yy = static_cast<io_t*>(p.y);
    uint4 cur_d[C::SPT], cur_u[C::SPT], cur_z[C::SPT];
    uint4 nxt_d[C::SPT], nxt_u[C::SPT], nxt_z[C::SPT];
    auto prefetch = [&](int64_t k, uint4(&vd)[C::SPT], uint4(&vu)[C::SPT], uint4(&vz)[C::SPT]) {
#pragma unroll
        for (int i = 0; i < C::SPT; ++i) {
            const int sidx = tid + i * NTH;
            const int cc = sidx % CH, seg = sidx / CH;
            const int64_t dd = d0 + cc;
            const bool ok = sidx < C::NSEG && dd < dim && k < nchunks;
            const int64_t row = (int64_t(b) * dim + (ok ? dd : 0)) * L;
            const int64_t t = k * T + seg * VEC;
            vd[i] = load_seg<C, VECIO>(dl + row, t, L, ok);
            vu[i] = load_seg<C, VECIO>(uu + row, t, L, ok);
            vz[i] = zz ? load_seg<C, VECIO>(zz + row, t, L, ok) : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    prefetch(0, cur_d, cur_u, cur_z);

    for (int64_t k = 0; k < nchunks; ++k) {
        const int64_t t0 = k * T;
        const int tlen = L - t0 < T ? int(L - t0) : T;

        // ---- phase A: B/C to fp32 shared memory, (dt, dt*u) per element ----
        float* sB = DIRECT ? reinterpret_cast<float*>(stageB(int(k))) : s.bf;
        float* sC = DIRECT ? reinterpret_cast<float*>(stageC(int(k))) : s.bf + T * NP;
        if (chunk_by_tma(k)) {
            if (!mbar_wait(&s.bar[k & 1], uint32_t(k >> 1) & 1u)) atomicOr(&g_scan_error, kErrWaitTimeout);
            if (!DIRECT) {
                const io_t* rb = reinterpret_cast<const io_t*>(stageB(int(k)));
                const io_t* rc = reinterpret_cast<const io_t*>(stageC(int(k)));
                for (int idx = tid; idx < T * NP; idx += NTH) {
                    const int t = idx / NP, n = idx % NP;
                    const bool ok = n < N;
                    sB[idx] = ok ? float(rb[t * N + n]) : 0.f;
                    sC[idx] = ok ? float(rc[t * N + n]) : 0.f;
                }
            }
        } else {
            for (int idx = tid; idx < T * NP; idx += NTH) {
                const int t = idx / NP, n = idx % NP;
                const bool ok = n < N && t < tlen;
                sB[idx] = ok ? float(Io<io_t>::load(Bg + (t0 + t) * N + n)) : 0.f;
                sC[idx] = ok ? float(Io<io_t>::load(Cg + (t0 + t) * N + n)) : 0.f;
            }
        }
#pragma unroll
        for (int i = 0; i < C::SPT; ++i) {
            const int sidx = tid + i * NTH;
            if (sidx >= C::NSEG) break;
            const int cc = sidx % CH, seg = sidx / CH;
            const int64_t dd = d0 + cc;
            const float bias = (dd < dim && p.delta_bias) ? __ldg(p.delta_bias + dd) : 0.f;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const int t = seg * VEC + e;
                float dt = Io<io_t>::get(cur_d[i], e) + bias;
                if (p.softplus) dt = C::ES == 2 ? softplus_fast(dt) : softplus_accurate(dt);
                float du = dt * Io<io_t>::get(cur_u[i], e);
                if (!(dd < dim && t < tlen)) dt = du = 0.f;
                s.du[t * CH + cc] = make_float4(dt, dt, du, du);
            }
        }
        prefetch(k + 1, nxt_d, nxt_u, nxt_z);
        __syncthreads();

        // ---- phase B: the recurrence ----
        auto run_steps = [&](auto full_tag) {
            constexpr bool FULL = decltype(full_tag)::value;
            const ulonglong2* du2 = reinterpret_cast<const ulonglong2*>(s.du);
            const ulonglong2* b2 = reinterpret_cast<const ulonglong2*>(sB);
            const ulonglong2* c2 = reinterpret_cast<const ulonglong2*>(sC);
            float4* yrow = reinterpret_cast<float4*>(s.y + tid * T);
            const int sw = yswz<T>(tid);
#pragma unroll 2
            for (int tt = 0; tt < T; tt += 4) {
                if (!FULL && tt >= tlen) break;
                float part[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int t = tt + j;
                    if (FULL || t < tlen) {
                        const ulonglong2 sd = du2[t * CH + c];  // (dt,dt), (du,du)
                        f32x2 acc = pack2(0.f, 0.f);
#pragma unroll
                        for (int q = 0; q < NQ; ++q) {
                            const ulonglong2 bq = b2[(t * NP + g * NPL) / 4 + q];
                            const ulonglong2 cq = c2[(t * NP + g * NPL) / 4 + q];
                            float x0, x1, x2, x3;
                            unpack2(mul2(sd.x, A2[2 * q]), x0, x1);
                            unpack2(mul2(sd.x, A2[2 * q + 1]), x2, x3);
                            const f32x2 a01 = pack2(ex2_approx(x0), ex2_approx(x1));
                            const f32x2 a23 = pack2(ex2_approx(x2), ex2_approx(x3));
                            h[2 * q] = fma2(a01, h[2 * q], mul2(sd.y, bq.x));
                            h[2 * q + 1] = fma2(a23, h[2 * q + 1], mul2(sd.y, bq.y));
                            acc = fma2(cq.x, h[2 * q], acc);
                            acc = fma2(cq.y, h[2 * q + 1], acc);
                        }
                        float lo, hi;
                        unpack2(acc, lo, hi);
                        part[j] = lo + hi;
                    } else {
                        part[j] = 0.f;
                    }
                }
                yrow[(tt / 4) ^ sw] = make_float4(part[0], part[1], part[2], part[3]);
            }
        };
        if (tlen == T)
            run_steps(std::integral_constant<bool, true>());
        else
            run_steps(std::integral_constant<bool, false>());
        __syncthreads();
        if (tid == 0 && k + 2 < nchunks && chunk_by_tma(k + 2)) {
            fence_proxy_async_smem();
            issue(k + 2);
        }

        // ---- phase C: reduce over state groups, skip, gate, store ----
#pragma unroll
        for (int i = 0; i < C::SPT; ++i) {
            const int sidx = tid + i * NTH;
            if (sidx >= C::NSEG) break;
            const int cc = sidx % CH, seg = sidx / CH;
            const int64_t dd = d0 + cc;
            if (dd >= dim || seg * VEC >= tlen) continue;
            float acc[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                const int r = cc * G + gg;
                const float4* yr = reinterpret_cast<const float4*>(s.y + r * T);
                const int sw = yswz<T>(r);
#pragma unroll
                for (int q = 0; q < VEC / 4; ++q) {
                    const float4 v = yr[(seg * (VEC / 4) + q) ^ sw];
                    acc[4 * q] += v.x;
                    acc[4 * q + 1] += v.y;
                    acc[4 * q + 2] += v.z;
                    acc[4 * q + 3] += v.w;
                }
            }
            const float Dd = p.D ? __ldg(p.D + dd) : 0.f;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                float v = fmaf(Dd, Io<io_t>::get(cur_u[i], e), acc[e]);
                if (zz) v *= silu_fast(Io<io_t>::get(cur_z[i], e));
                acc[e] = v;
            }
            store_seg<C, VECIO>(yy + (int64_t(b) * dim + dd) * L, t0 + seg * VEC, L, acc);
        }
#pragma unroll
        for (int i = 0; i < C::SPT; ++i) {
            cur_d[i] = nxt_d[i];
            cur_u[i] = nxt_u[i];
            cur_z[i] = nxt_z[i];
        }
    }

    if (chain_ok && p.last_state) {
        float* out = p.last_state + (int64_t(b) * dim + d) * N;
#pragma unroll
        for (int q = 0; q < 2 * NQ; ++q) {
            float v[2];
            unpack2(h[q], v[0], v[1]);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int n = g * NPL + 2 * q + e;
                if (n < N) out[n] = v[e];
            }
        }
    }
}

template <typename io_t, int NPL, int G, int CH, int T>
cudaError_t launch_cfg(const ScanArgs& a, cudaStream_t stream) {
    using C = Cfg<io_t, NPL, G, CH, T>;
    const size_t es = sizeof(io_t);
    auto al16 = [](const void* q) { return q == nullptr || (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
    const bool vecio = al16(a.u) && al16(a.delta) && al16(a.z) && al16(a.y) &&
                       (a.seqlen * int64_t(es)) % 16 == 0;
    const bool direct = es == 4 && a.dstate == C::NP;
    const int tma_ok = al16(a.B) && al16(a.C) && (a.seqlen * a.dstate * int64_t(es)) % 16 == 0 &&
                       (int64_t(T) * a.dstate * int64_t(es)) % 16 == 0;
    const int64_t dblocks = (a.dim + CH - 1) / CH;
    const int64_t blocks = dblocks * a.batch;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;

    auto go = [&](auto kern, size_t smem) -> cudaError_t {
        cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               int(smem));
        if (err != cudaSuccess) return err;
        kern<<<unsigned(blocks), C::NTH, smem, stream>>>(a, int(dblocks), tma_ok);
        return cudaGetLastError();
    };
    if constexpr (sizeof(io_t) == 4) {
        if (direct) {
            if (vecio) return go(scan_fwd_kernel<io_t, NPL, G, CH, T, true, true>, C::kSmemDirect);
            return go(scan_fwd_kernel<io_t, NPL, G, CH, T, false, true>, C::kSmemDirect);
        }
    }
    if (vecio) return go(scan_fwd_kernel<io_t, NPL, G, CH, T, true, false>, C::kSmem);
    return go(scan_fwd_kernel<io_t, NPL, G, CH, T, false, false>, C::kSmem);
}

template <typename io_t>
cudaError_t dispatch(const ScanArgs& a, cudaStream_t stream) {
    const int N = a.dstate;
    if (N <= 4) return launch_cfg<io_t, 4, 1, 64, 8>(a, stream);
    if (N <= 8) return launch_cfg<io_t, 4, 2, 32, 16>(a, stream);
    if (N <= 16) return launch_cfg<io_t, 4, 4, 16, 32>(a, stream);
    if (N <= 32) return launch_cfg<io_t, 4, 8, 8, 32>(a, stream);
    if (N <= 64) return launch_cfg<io_t, 4, 16, 4, 16>(a, stream);
    if (N <= 128) return launch_cfg<io_t, 4, 32, 2, 16>(a, stream);
    return launch_cfg<io_t, 8, 32, 2, 8>(a, stream);
}

}  // namespace

cudaError_t launch_scan_fwd(const ScanArgs& a, bool bf16, cudaStream_t stream) {
    return bf16 ? dispatch<__nv_bfloat16>(a, stream) : dispatch<float>(a, stream);
}

cudaError_t read_and_clear_device_error(unsigned int* word, cudaStream_t stream) {
    cudaError_t err = cudaStreamSynchronize(stream);
    if (err != cudaSuccess) return err;
    err = cudaMemcpyFromSymbol(word, g_scan_error, sizeof(unsigned int));
    if (err != cudaSuccess) return err;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_scan_error, &zero, sizeof(unsigned int));
}

}  // namespace mamba
