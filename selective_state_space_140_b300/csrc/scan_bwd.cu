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
//                     and form every gradient of the step (the fp64 oracle
//                     writes the same chain rule out).
//
// Few chains over a long sequence split it along time: a summary pass gives
// each (chain, segment) its zero-start end state, sum of dt and zero-start
// adjoint leaving to the left; a carry pass passes states forwards and
// adjoints backwards across segments (both decay by exp(A * sum of dt over
// the segment)); the full pass then runs every segment from its entering
// state and adjoint, all segments in parallel.
//
// Latency: every chunk's raw inputs (delta, u, dout, z, B, C and the
// checkpoint) are fetched into registers one chunk ahead, so the loads of
// chunk k-1 are in flight while chunk k computes; loops have compile-time trip
// counts (a short last chunk is padded with dt = u = dout = B = C = 0 steps,
// which leave the state and every gradient unchanged).  The values of one
// element (a chain and a step) stay in the registers of the thread that
// loaded them; only what other threads read goes through shared memory.
//
// B, C, A_log, D and the bias are shared by many chains, so their gradients
// are sums.  dC[t,n] = sum_c dy_ct h_ctn and dB[t,n] = sum_c dt_ct u_ct g_ctn
// are formed once per chunk from the states (then the adjoints, which the
// backward sweep writes over the states it has used) in shared memory -- a
// small product over the CTA's chains per step -- and added to the fp32
// outputs with 16-byte atomics; dA_log, dD and the bias gradient accumulate
// over the whole sequence and are added once at the end.
#include <cstdlib>

#include "scan_bwd.cuh"
#include "scratch_pool.cuh"

namespace mamba {
namespace {

constexpr int kBT = 16;     // steps per chunk
constexpr int kBNTH = 64;   // threads per CTA

template <typename io_t, int NPL_, int G_>
struct BwdCfg {
    static constexpr int NPL = NPL_, G = G_, T = kBT, NTH = kBNTH;
    static constexpr int CH = NTH / G;        // chains per CTA
    static constexpr int NP = NPL * G;        // states per chain, padded
    static constexpr int NQ = NPL / 4;        // float4 per thread per step
    static constexpr int kE = T * CH;         // elements (chain, step) per chunk
    // elements per thread: EPT consecutive steps of one chain
    static constexpr int EPT = (kE + NTH - 1) / NTH;
    static constexpr int BPT = (T * NP + NTH - 1) / NTH;  // B (and C) values per thread
    // [t][chain] fields use a padded row so that the element role (EPT
    // consecutive steps per thread) and the chain role both access them
    // without bank conflicts: kS = CH + 2 (or + 4) makes EPT * kS an odd
    // multiple of 32 / (T / EPT) modulo 32.
    static constexpr int kS = ((CH + 2) / 2) % 2 == 1 ? CH + 2 : CH + 4;
    static constexpr int kF = T * kS;
    // shared memory (floats)
    static constexpr int oDt = 0, oU = kF, oDy = 2 * kF;
    static constexpr int oGu = 3 * kF, oGdt = 4 * kF;   // reduced sum_n g B, sum_n g (...)
    static constexpr int oYs = 5 * kF;                   // C.h
    static constexpr int oDe = 6 * kF;  // dt in the decay: +inf at a document start (reset only)
    static constexpr int oB = 7 * kF, oC = oB + T * NP;
    static constexpr int oH = oC + T * NP;  // [T][NQ][NTH] float4: states, then adjoints
    static constexpr int kFloats = oH + T * NQ * NTH * 4;
    static constexpr size_t kSmem = size_t(kFloats) * 4;
    static_assert(NPL % 4 == 0, "states per lane in whole float4");
    static_assert(T % EPT == 0, "a thread's elements stay within one chain");
    static_assert(oH % 4 == 0, "float4 state tiles");
};

struct BwdArgs : ScanBwdArgs {
    float* ckpt;  // [batch * dim][nchunks][N] scratch: state at each chunk start
    float* dh0 = nullptr;  // [batch * dim][N] or nullptr: gradient of f.h0
    // time split (nseg > 1): segment s covers chunks [s * seg_chunks, (s+1) * seg_chunks)
    int nseg = 1, seg_chunks = 0;
    float* hseg = nullptr;  // [chains][nseg][N]: summary: zero-start end state; main: state entering
    float* gseg = nullptr;  // [chains][nseg][N]: summary: zero-start adjoint leaving to the left;
                            //                    main: Abar g entering from the right
    float* sdt = nullptr;   // [chains][nseg]: sum of dt over the segment
};

constexpr int kBwdFull = 0, kBwdSummary = 1;

// One chunk's raw inputs as fetched (converted to float only when staged, so
// that no instruction waits on the loads before the chunk is used).
template <typename io_t, int NPL, int G>
struct Raw {
    using C = BwdCfg<io_t, NPL, G>;
    io_t dl[C::EPT], u[C::EPT], go[C::EPT], z[C::EPT];
    io_t B[C::BPT], Cc[C::BPT];
    float hs[NPL];  // checkpoint: the state at the chunk's start
    unsigned char rs[C::EPT];  // document starts (when a reset mask is given)
};

template <typename io_t>
__device__ __forceinline__ float to_f(io_t v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// Issue the loads of chunk k (REV: everything the reverse phase needs; else
// only delta, u and B).  Out-of-range elements read as zero.
template <typename io_t, int NPL, int G, bool REV, bool EX>
__device__ __forceinline__ void fetch(const BwdArgs& a, Raw<io_t, NPL, G>& r, int b, int64_t d0,
                                      int64_t k, int tid, const float* ck, bool chain_ok, int g) {
    using C = BwdCfg<io_t, NPL, G>;
    const ScanArgs& p = a.f;
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
        if constexpr (EX) r.rs[j] = (ok && p.reset) ? __ldg(p.reset + int64_t(b) * L + t0 + t) : 0;
        if constexpr (REV) {
            r.go[j] = ok ? __ldg(static_cast<const io_t*>(a.dout) + idx) : zero;
            r.z[j] = (ok && p.z) ? __ldg(static_cast<const io_t*>(p.z) + idx) : zero;
        }
    }
    const io_t* Bg = static_cast<const io_t*>(p.B) + int64_t(b) * L * N;
    const io_t* Cg = static_cast<const io_t*>(p.C) + int64_t(b) * L * N;
#pragma unroll
    for (int j = 0; j < C::BPT; ++j) {
        const int e = tid + j * C::NTH;
        const int t = e / C::NP, n = e % C::NP;
        const bool ok = e < C::T * C::NP && n < N && t0 + t < L;
        const int64_t off = ok ? (t0 + t) * N + n : 0;
        r.B[j] = ok ? __ldg(Bg + off) : zero;
        if constexpr (REV) r.Cc[j] = ok ? __ldg(Cg + off) : zero;
    }
    if constexpr (REV) {
#pragma unroll
        for (int i = 0; i < NPL; ++i)
            r.hs[i] = (chain_ok && g * NPL + i < N) ? ck[k * N + g * NPL + i] : 0.f;
    }
}

// dst[t][n0 .. n0+3] of chunk rows (b, t0 + t) += sum over the CTA's chains of
// w[t][c] * S[t][c][n0 .. n0+3], for every step and state quad of the chunk
// (S: the [T][NQ][NTH] float4 tile; w: a [t][chain] field or dt * u).  At odd
// steps chain c's column of the tile is that of chain c ^ 1 (tile_col), so
// the lanes of a quarter-warp -- two steps, the same chains -- read different
// banks while the chain loop runs in a fixed order with constant offsets.
template <typename io_t, int NPL, int G, bool DTU>
__device__ __forceinline__ void chain_product(const float* sm, const float4* S, int wfield,
                                              float* dst, int tlen, int N, bool vec_red, int tid) {
    using C = BwdCfg<io_t, NPL, G>;
    constexpr int NP4 = C::NP / 4;
    for (int o = tid; o < C::T * NP4; o += C::NTH) {
        const int t = o / NP4, n0 = (o % NP4) * 4;
        if (t >= tlen || n0 >= N) continue;
        const int g = n0 / NPL, q = (n0 % NPL) / 4;
        const int sw = (t & 1) * G;
        // chain c at step t: column (c ^ (t & 1)) * G + g, i.e. c * G + g + sw
        // for even c and c * G + g - sw for odd c
        const float4* se = S + (t * C::NQ + q) * C::NTH + g + sw;
        const float4* so = S + (t * C::NQ + q) * C::NTH + g - sw;
        const float* w0 = sm + (DTU ? C::oDt : wfield) + t * C::kS;
        const float* w1 = sm + C::oU + t * C::kS;
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int c = 0; c < C::CH; ++c) {
            const float w = DTU ? w0[c] * w1[c] : w0[c];
            const float4 x = (c & 1) ? so[c * G] : se[c * G];
            sum.x = fmaf(w, x.x, sum.x);
            sum.y = fmaf(w, x.y, sum.y);
            sum.z = fmaf(w, x.z, sum.z);
            sum.w = fmaf(w, x.w, sum.w);
        }
        float* out = dst + t * N + n0;
        if (vec_red) {
            atomicAdd(reinterpret_cast<float4*>(out), sum);
        } else {
            const float vals[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (n0 + e < N) atomicAdd(out + e, vals[e]);
        }
    }
}

// MODE kBwdFull: gradients of the segment's elements (the whole sequence when
// unsplit).  MODE kBwdSummary: the segment's zero-start end state, its sum of
// dt and its zero-start adjoint leaving to the left (no gradients), for the
// carry pass of a time-split backward.
// EX: h0, document resets and dh0 are handled (compiled separately so that the
// plain backward's code is unchanged by them).
template <typename io_t, int NPL, int G, int UA, int MODE, bool EX>
__global__ void __launch_bounds__(kBNTH, NPL == 4 ? 8 : 1) scan_bwd_kernel(const BwdArgs a, const int dblocks,
                                                         const bool vec_red) {
    using C = BwdCfg<io_t, NPL, G>;
    constexpr int T = C::T, NTH = C::NTH, CH = C::CH, NP = C::NP, NQ = C::NQ, S = C::kS;
    constexpr int EPT = C::EPT;
    extern __shared__ __align__(16) float sm[];
    float4* sH = reinterpret_cast<float4*>(sm + C::oH);

    const ScanArgs& p = a.f;
    const int64_t L = p.seqlen, dim = p.dim;
    const int N = p.dstate;
    // blockIdx.x = (b * dblocks + channel block) * nseg + time segment
    const int seg = blockIdx.x % a.nseg;
    const int cblk = blockIdx.x / a.nseg;
    const int b = cblk / dblocks;
    const int64_t d0 = int64_t(cblk % dblocks) * CH;
    // recurrence role: chain c, states g * NPL ..; element role: chain ce, steps te0 ..
    const int tid = threadIdx.x, c = tid / G, g = tid % G;
    // this thread's column of the state / adjoint tile at step t: its own at
    // even steps, chain c ^ 1's at odd steps (see chain_product)
    auto tile_col = [&](int t) { return (t & 1) ? (tid ^ G) : tid; };
    const int e0 = tid * EPT, ce = e0 / T, te0 = e0 % T;
    const bool e_live = e0 < C::kE && d0 + ce < dim;  // this thread owns real elements
    const int64_t de = e_live ? d0 + ce : 0;
    const float e_bias = (e_live && p.delta_bias) ? __ldg(p.delta_bias + de) : 0.f;
    const float e_D = (e_live && p.D) ? __ldg(p.D + de) : 0.f;
    const int64_t d = d0 + c;
    const bool chain_ok = d < dim;
    const int64_t chain = int64_t(b) * dim + (chain_ok ? d : 0);
    const int64_t nchunks = (L + T - 1) / T;
    float* ck = a.ckpt + chain * nchunks * N;
    const int64_t kbeg = a.nseg > 1 ? int64_t(seg) * a.seg_chunks : 0;
    const int64_t kend = a.nseg > 1 ? (kbeg + a.seg_chunks < nchunks ? kbeg + a.seg_chunks : nchunks)
                                    : nchunks;
    float* hsg = a.nseg > 1 ? a.hseg + (chain * a.nseg + seg) * N : nullptr;
    float* gsg = a.nseg > 1 ? a.gseg + (chain * a.nseg + seg) * N : nullptr;

    float A[NPL], A2[NPL], h[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        const int n = g * NPL + i;
        A[i] = (chain_ok && n < N) ? -expf(__ldg(p.A_log + d * N + n)) : 0.f;
        // at most -1e-30, so that a document start's infinite decay step gives
        // Abar = 0 exactly (and padded states, with B = C = 0, stay zero)
        A2[i] = EX ? fminf(A[i] * kLog2e, -1e-30f) : A[i] * kLog2e;
        // the first segment starts from h0 (or zero), a later one of a split
        // from the carried state
        float h_in = 0.f;
        if (MODE == kBwdFull && chain_ok && n < N)
            h_in = hsg ? hsg[n] : ((EX && p.h0) ? p.h0[chain * N + n] : 0.f);
        h[i] = h_in;
    }
    // the same as pairs of states, for the packed f32x2 arithmetic of the reverse phase
    constexpr int NH = NPL / 2;
    f32x2 Ap[NH], A2p[NH];
#pragma unroll
    for (int q = 0; q < NH; ++q) {
        Ap[q] = pack2(A[2 * q], A[2 * q + 1]);
        A2p[q] = pack2(A2[2 * q], A2[2 * q + 1]);
    }
    float dtsum = 0.f;  // summary: sum of the decay steps over the segment
    const bool has_reset = EX && p.reset != nullptr;
    constexpr float kDocStart = __builtin_inff();  // decay step of a document's first token

    // dt (and softplus') of element j of this thread in chunk k; zero past the data
    auto step_of = [&](float raw_delta, int64_t k, int j, float& sp) {
        const bool ok = e_live && k * T + te0 + j < L;
        const float raw = raw_delta + e_bias;
        float dt = raw;
        sp = 1.f;
        if (p.softplus) {
            dt = sizeof(io_t) == 2 ? softplus_fast(raw) : softplus_accurate(raw);
            sp = rcp_approx(1.f + ex2_approx(-raw * kLog2e));
        }
        if (!ok) dt = sp = 0.f;
        return dt;
    };

    Raw<io_t, NPL, G> r;
    // ---------------- forward phase: checkpoints ----------------
    if (kbeg < kend) fetch<io_t, NPL, G, false, EX>(a, r, b, d0, kbeg, tid, ck, chain_ok, g);
    for (int64_t k = kbeg; k < kend; ++k) {
        __syncthreads();
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
            float sp;
            const float dt = step_of(to_f(r.dl[j]), k, j, sp);
            if (e0 + j < C::kE) {
                sm[C::oDt + (te0 + j) * S + ce] = dt;
                sm[C::oU + (te0 + j) * S + ce] = dt * to_f(r.u[j]);  // dt u
                if (has_reset) sm[C::oDe + (te0 + j) * S + ce] = r.rs[j] ? kDocStart : dt;
            }
        }
#pragma unroll
        for (int j = 0; j < C::BPT; ++j)
            if (tid + j * NTH < T * NP) sm[C::oB + tid + j * NTH] = to_f(r.B[j]);
        if (MODE == kBwdFull && chain_ok) {
#pragma unroll
            for (int i = 0; i < NPL; ++i)
                if (g * NPL + i < N) ck[k * N + g * NPL + i] = h[i];
        }
        __syncthreads();
        if (k + 1 < kend)
            fetch<io_t, NPL, G, false, EX>(a, r, b, d0, k + 1, tid, ck, chain_ok, g);
        else
            fetch<io_t, NPL, G, true, EX>(a, r, b, d0, k, tid, ck, chain_ok, g);
#pragma unroll
        for (int t = 0; t < T; ++t) {
            const float dt = sm[C::oDt + t * S + c], du = sm[C::oU + t * S + c];
            const float de = has_reset ? sm[C::oDe + t * S + c] : dt;
            if (MODE == kBwdSummary) dtsum += de;
#pragma unroll
            for (int i = 0; i < NPL; ++i)
                h[i] = fmaf(ex2_approx(de * A2[i]), h[i], du * sm[C::oB + t * NP + g * NPL + i]);
        }
    }
    if (MODE == kBwdSummary && chain_ok) {
#pragma unroll
        for (int i = 0; i < NPL; ++i)
            if (g * NPL + i < N) hsg[g * NPL + i] = h[i];
        if (g == 0) a.sdt[chain * a.nseg + seg] = dtsum;
    }

    // ---------------- reverse phase ----------------
    float gc[NPL], dA[NPL];  // Abar_{t+1} g_{t+1}; sum of g dt Abar h_{t-1}
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        // The adjoint entering the last step from the right is the gradient on
        // the final state (zero without one); a split's segments start from
        // the carried adjoint, which holds it for the last segment.
        const int n = g * NPL + i;
        float gin = 0.f;
        if (MODE == kBwdFull && chain_ok && n < N) {
            if (gsg)
                gin = gsg[n];
            else if (EX && a.dlast)
                gin = a.dlast[chain * N + n];
        }
        gc[i] = gin;
        dA[i] = 0.f;
    }
    float accD = 0.f, accB = 0.f;  // this thread's elements: sums of dy u and ddelta
    for (int64_t k = kend - 1; k >= kbeg; --k) {
        const int64_t t0 = k * T;
        const int tlen = L - t0 < T ? int(L - t0) : T;
        float* dBg = a.dB + (int64_t(b) * L + t0) * N;
        float* dCg = a.dC + (int64_t(b) * L + t0) * N;
        __syncthreads();
        // stage chunk k: dt and u for every thread, the rest stays in registers
        float e_sp[EPT], e_go[EPT], e_z[EPT], hs[NPL];
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
            const float dt = step_of(to_f(r.dl[j]), k, j, e_sp[j]);
            e_go[j] = to_f(r.go[j]);
            e_z[j] = to_f(r.z[j]);
            if (e0 + j < C::kE) {
                sm[C::oDt + (te0 + j) * S + ce] = dt;
                sm[C::oU + (te0 + j) * S + ce] = to_f(r.u[j]);
                if (has_reset) sm[C::oDe + (te0 + j) * S + ce] = r.rs[j] ? kDocStart : dt;
            }
        }
#pragma unroll
        for (int j = 0; j < C::BPT; ++j)
            if (tid + j * NTH < T * NP) {
                sm[C::oB + tid + j * NTH] = to_f(r.B[j]);
                sm[C::oC + tid + j * NTH] = to_f(r.Cc[j]);
            }
#pragma unroll
        for (int i = 0; i < NPL; ++i) hs[i] = r.hs[i];
        __syncthreads();
        if (k > kbeg) fetch<io_t, NPL, G, true, EX>(a, r, b, d0, k - 1, tid, ck, chain_ok, g);
        if constexpr (MODE == kBwdSummary) {
            // dy for every element, then the adjoint alone (no states needed)
#pragma unroll
            for (int j = 0; j < EPT; ++j) {
                if (e0 + j >= C::kE) continue;
                const int s = (te0 + j) * S + ce;
                float dy = e_go[j];
                if (p.z) {
                    const float z = e_z[j];
                    dy = e_go[j] * (z * rcp_approx(1.f + ex2_approx(-z * kLog2e)));
                }
                sm[C::oDy + s] = dy;
            }
            __syncthreads();
#pragma unroll UA
            for (int t = T - 1; t >= 0; --t) {
                const int s = t * S + c;
                const float dy = sm[C::oDy + s];
                const float de = has_reset ? sm[C::oDe + s] : sm[C::oDt + s];
#pragma unroll
                for (int i = 0; i < NPL; ++i) {
                    const float gn = fmaf(dy, sm[C::oC + t * NP + g * NPL + i], gc[i]);
                    gc[i] = ex2_approx(de * A2[i]) * gn;
                }
            }
            continue;
        }

        // recompute the chunk's states into shared memory; C.h summed over the
        // chain's lanes by a butterfly per step
        {
            // states in pairs (packed f32x2), B and C of the lane's states as float4
            f32x2 hh[NH];
#pragma unroll
            for (int q = 0; q < NH; ++q) hh[q] = pack2(hs[2 * q], hs[2 * q + 1]);
#pragma unroll
            for (int t = 0; t < T; ++t) {
                const float dt = sm[C::oDt + t * S + c];
                const float du = dt * sm[C::oU + t * S + c];
                const float de = has_reset ? sm[C::oDe + t * S + c] : dt;
                const float4* Bt = reinterpret_cast<const float4*>(sm + C::oB + t * NP + g * NPL);
                const float4* Ct = reinterpret_cast<const float4*>(sm + C::oC + t * NP + g * NPL);
                const f32x2 des = pack2(de, de), dus = pack2(du, du);
                f32x2 acc2 = pack2(0.f, 0.f);
#pragma unroll
                for (int v = 0; v < NQ; ++v) {
                    const float4 bv = Bt[v], cv = Ct[v];
                    const f32x2 bq[2] = {pack2(bv.x, bv.y), pack2(bv.z, bv.w)};
                    const f32x2 cq[2] = {pack2(cv.x, cv.y), pack2(cv.z, cv.w)};
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int q = 2 * v + e;
                        float x0, x1;
                        unpack2(mul2(des, A2p[q]), x0, x1);
                        hh[q] = fma2(pack2(ex2_approx(x0), ex2_approx(x1)), hh[q], mul2(dus, bq[e]));
                        acc2 = fma2(cq[e], hh[q], acc2);
                    }
                }
                float acc_lo, acc_hi;
                unpack2(acc2, acc_lo, acc_hi);
                float acc = acc_lo + acc_hi;
#pragma unroll
                for (int v = 0; v < NQ; ++v) {
                    float h0v, h1v, h2v, h3v;
                    unpack2(hh[2 * v], h0v, h1v);
                    unpack2(hh[2 * v + 1], h2v, h3v);
                    sH[(t * NQ + v) * NTH + tile_col(t)] = make_float4(h0v, h1v, h2v, h3v);
                }
#pragma unroll
                for (int off = G / 2; off > 0; off /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, off);
                if (g == 0) sm[C::oYs + t * S + c] = acc;
            }
        }
        __syncthreads();

        // this thread's elements: y = C.h + D u, the gate's gradient, dy
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
            if (e0 + j >= C::kE) continue;
            const int t = te0 + j, s = t * S + ce;
            const float y = fmaf(e_D, sm[C::oU + s], sm[C::oYs + s]);
            const float go = e_go[j];
            float dy = go;
            if (p.z) {
                const float z = e_z[j];
                const float sg = rcp_approx(1.f + ex2_approx(-z * kLog2e));
                if (e_live && t < tlen)
                    Io<io_t>::store(static_cast<io_t*>(a.dz) + (int64_t(b) * dim + de) * L + t0 + t,
                                    go * y * (sg * (1.f + z * (1.f - sg))));
                dy = go * (z * sg);
            }
            sm[C::oDy + s] = dy;
        }
        __syncthreads();

        // dC of the chunk from the states
        chain_product<io_t, NPL, G, false>(sm, sH, C::oDy, dCg, tlen, N, vec_red, tid);
        __syncthreads();

        // adjoint, backwards through the chunk; g_t replaces h_t in the tile
        // once step t has read it (step t-1 reads only h_{t-1} and h_{t-2})
        // packed f32x2 over pairs of states; gc and dA as pairs during the sweep
        f32x2 gcp[NH], dAp[NH];
#pragma unroll
        for (int q = 0; q < NH; ++q) {
            gcp[q] = pack2(gc[2 * q], gc[2 * q + 1]);
            dAp[q] = pack2(dA[2 * q], dA[2 * q + 1]);
        }
#pragma unroll UA
        for (int t = T - 1; t >= 0; --t) {
            const int s = t * S + c;
            const float dy = sm[C::oDy + s], dt = sm[C::oDt + s], u = sm[C::oU + s];
            const float de = has_reset ? sm[C::oDe + s] : dt;  // Abar = 0 at a document start
            const float4* Bt = reinterpret_cast<const float4*>(sm + C::oB + t * NP + g * NPL);
            const float4* Ct = reinterpret_cast<const float4*>(sm + C::oC + t * NP + g * NPL);
            const f32x2 des = pack2(de, de), dys = pack2(dy, dy), dts = pack2(dt, dt);
            f32x2 gu2 = pack2(0.f, 0.f), gd2 = pack2(0.f, 0.f);
#pragma unroll
            for (int v = 0; v < NQ; ++v) {
                const float4 hv = t > 0 ? sH[((t - 1) * NQ + v) * NTH + tile_col(t - 1)]
                                        : make_float4(hs[4 * v], hs[4 * v + 1], hs[4 * v + 2],
                                                      hs[4 * v + 3]);
                const float4 bv = Bt[v], cv = Ct[v];
                const f32x2 hq[2] = {pack2(hv.x, hv.y), pack2(hv.z, hv.w)};
                const f32x2 bq[2] = {pack2(bv.x, bv.y), pack2(bv.z, bv.w)};
                const f32x2 cq[2] = {pack2(cv.x, cv.y), pack2(cv.z, cv.w)};
                f32x2 gq[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int q = 2 * v + e;
                    float x0, x1;
                    unpack2(mul2(des, A2p[q]), x0, x1);
                    const f32x2 ab = pack2(ex2_approx(x0), ex2_approx(x1));
                    const f32x2 gn = fma2(dys, cq[e], gcp[q]);
                    const f32x2 w = mul2(gn, mul2(ab, hq[e]));
                    gq[e] = gn;
                    gu2 = fma2(gn, bq[e], gu2);
                    gd2 = fma2(Ap[q], w, gd2);
                    dAp[q] = fma2(dts, w, dAp[q]);
                    gcp[q] = mul2(ab, gn);
                }
                float g0, g1, g2, g3;
                unpack2(gq[0], g0, g1);
                unpack2(gq[1], g2, g3);
                sH[(t * NQ + v) * NTH + tile_col(t)] = make_float4(g0, g1, g2, g3);
            }
            float gu_lo, gu_hi, gd_lo, gd_hi;
            unpack2(gu2, gu_lo, gu_hi);
            unpack2(gd2, gd_lo, gd_hi);
            float gu = gu_lo + gu_hi, gd = gd_lo + gd_hi;
            gd = fmaf(u, gu, gd);  // sum_n g (A Abar h_{t-1} + u B)
            if constexpr (G >= 2) {
                // Both sums over the chain's G lanes at once: in the first
                // round lane g keeps gu (g even) or gd (g odd) and sends the
                // other to its partner; the remaining rounds reduce the one
                // kept value, which lane 0 (gu) and lane 1 (gd) then store.
                const bool odd = g & 1;
                float v = (odd ? gd : gu) + __shfl_xor_sync(0xffffffffu, odd ? gu : gd, 1);
#pragma unroll
                for (int off = 2; off < G; off *= 2) v += __shfl_xor_sync(0xffffffffu, v, off);
                if (g < 2) sm[(odd ? C::oGdt : C::oGu) + s] = v;
            } else {
                sm[C::oGu + s] = gu;
                sm[C::oGdt + s] = gd;
            }
        }
#pragma unroll
        for (int q = 0; q < NH; ++q) {
            unpack2(gcp[q], gc[2 * q], gc[2 * q + 1]);
            unpack2(dAp[q], dA[2 * q], dA[2 * q + 1]);
        }
        __syncthreads();

        // dB of the chunk from the adjoints
        chain_product<io_t, NPL, G, true>(sm, sH, 0, dBg, tlen, N, vec_red, tid);

        // this thread's elements: du, ddelta, and the sums for dD and the bias
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
            const int t = te0 + j;
            if (!(e_live && t < tlen)) continue;
            const int s = t * S + ce;
            const int64_t idx = (int64_t(b) * dim + de) * L + t0 + t;
            const float dy = sm[C::oDy + s];
            const float du = fmaf(sm[C::oDt + s], sm[C::oGu + s], dy * e_D);
            const float dr = sm[C::oGdt + s] * e_sp[j];
            Io<io_t>::store(static_cast<io_t*>(a.du) + idx, du);
            Io<io_t>::store(static_cast<io_t*>(a.ddelta) + idx, dr);
            accD = fmaf(dy, sm[C::oU + s], accD);
            accB += dr;
        }
    }

    if constexpr (MODE == kBwdSummary) {
        if (chain_ok) {
#pragma unroll
            for (int i = 0; i < NPL; ++i)
                if (g * NPL + i < N) gsg[g * NPL + i] = gc[i];
        }
        return;
    }
    // the adjoint carried out of step 0 is the gradient of h0
    if (EX && a.dh0 && seg == 0 && chain_ok) {
#pragma unroll
        for (int i = 0; i < NPL; ++i)
            if (g * NPL + i < N) a.dh0[chain * N + g * NPL + i] = gc[i];
    }
    // dA_log = dA * A (A = -exp(A_log)); dD and the bias gradient per chain
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        const int n = g * NPL + i;
        if (chain_ok && n < N) atomicAdd(a.dA_log + d * N + n, dA[i] * A[i]);
    }
    constexpr int R = T / EPT;  // threads that share a chain's elements
#pragma unroll
    for (int off = R / 2; off > 0; off /= 2) {
        accD += __shfl_xor_sync(0xffffffffu, accD, off);
        accB += __shfl_xor_sync(0xffffffffu, accB, off);
    }
    if (e_live && tid % R == 0) {
        if (a.dD) atomicAdd(a.dD + de, accD);
        if (a.ddelta_bias) atomicAdd(a.ddelta_bias + de, accB);
    }
}

// Carry pass of a time-split backward, one thread per (chain, state).  With
// P(s) = exp(A * sum of dt over s), the product of the segment's decays:
//   forward: the state entering s + 1 is P(s) times the state entering s plus
//            the zero-start end state of s (hseg becomes the entering states);
//   adjoint: Abar g entering s from the right is a(s + 1) + P(s + 1) times the
//            value entering s + 1, a(s) the zero-start adjoint leaving s to the
//            left; for the last segment it is the gradient on the final state
//            (or zero) (gseg becomes the entering values).
__global__ void __launch_bounds__(256) bwd_carry_kernel(const float* A_log, const float* h0,
                                                        const float* dlast, float* hseg, float* gseg,
                                                        const float* sdt, int64_t chains,
                                                        int64_t dim, int N, int nseg) {
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= chains * N) return;
    const int64_t chain = i / N;
    const int n = int(i % N);
    const float A2 = fminf(-expf(__ldg(A_log + (chain % dim) * N + n)) * kLog2e, -1e-30f);
    float* hs = hseg + chain * nseg * N + n;
    float* gs = gseg + chain * nseg * N + n;
    const float* sd = sdt + chain * nseg;
    float H = h0 ? h0[i] : 0.f;  // the state entering segment 0
    for (int s = 0; s < nseg; ++s) {
        const float e = hs[int64_t(s) * N];
        hs[int64_t(s) * N] = H;
        H = fmaf(ex2_approx(A2 * sd[s]), H, e);
    }
    float Gv = dlast ? dlast[i] : 0.f;  // the gradient on the final state enters the last segment
    for (int s = nseg - 1; s >= 0; --s) {
        const float e = gs[int64_t(s) * N];
        gs[int64_t(s) * N] = Gv;
        Gv = fmaf(ex2_approx(A2 * sd[s]), Gv, e);
    }
}

template <typename io_t, int NPL, int G, int UA, bool EX>
cudaError_t launch_bwd_impl(const BwdArgs& a0, bool vec_red, cudaStream_t stream) {
    using C = BwdCfg<io_t, NPL, G>;
    const int64_t dblocks = (a0.f.dim + C::CH - 1) / C::CH;
    const int64_t ctas = dblocks * a0.f.batch;
    const int64_t nchunks = (a0.f.seqlen + kBT - 1) / kBT;
    // Few CTAs for the GPU (under two per SM) and a long sequence: split the
    // sequence into segments (at least 32 chunks each), about two waves of 7
    // CTAs per SM (measured on the 1 x 1536 x 131072 layer: 11.7 ms against
    // 12.6 ms with one wave; with two or more CTAs per SM unsplit a split was
    // slower: 9.6 vs 7.2 ms at 2 x 2048 x 8192, N 64).  MAMBA_BWD_SEGMENTS
    // forces a segment count.
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t nseg = 1;
    const char* env = getenv("MAMBA_BWD_SEGMENTS");
    if (env && atoi(env) > 0) {
        nseg = atoi(env);
    } else if (ctas < 2 * int64_t(sms) && nchunks >= 64) {
        nseg = (14 * int64_t(sms) + ctas - 1) / ctas;
        if (nseg > nchunks / 32) nseg = nchunks / 32;
    }
    if (nseg > nchunks) nseg = nchunks;
    if (nseg < 1) nseg = 1;
    const int64_t seg_chunks = (nchunks + nseg - 1) / nseg;
    nseg = (nchunks + seg_chunks - 1) / seg_chunks;
    if (ctas * nseg > 0x7fffffff) return cudaErrorInvalidConfiguration;

    cudaError_t err = cudaSuccess;
    BwdArgs a = a0;
    a.nseg = int(nseg);
    a.seg_chunks = int(seg_chunks);
    void* seg_mem = nullptr;
    if (nseg > 1) {
        const int64_t chains = a.f.batch * a.f.dim;
        const size_t nst = size_t(chains) * nseg * a.f.dstate;
        if ((err = scratch_alloc(&seg_mem, (2 * nst + size_t(chains) * nseg) * sizeof(float),
                                   stream)) != cudaSuccess)
            return err;
        a.hseg = static_cast<float*>(seg_mem);
        a.gseg = a.hseg + nst;
        a.sdt = a.gseg + nst;
        err = cudaFuncSetAttribute(scan_bwd_kernel<io_t, NPL, G, UA, kBwdSummary, EX>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::kSmem));
        if (err == cudaSuccess) {
            scan_bwd_kernel<io_t, NPL, G, UA, kBwdSummary, EX>
                <<<unsigned(ctas * nseg), C::NTH, C::kSmem, stream>>>(a, int(dblocks), vec_red);
            err = cudaGetLastError();
        }
        if (err == cudaSuccess) {
            const int64_t n = chains * a.f.dstate;
            bwd_carry_kernel<<<unsigned((n + 255) / 256), 256, 0, stream>>>(
                a.f.A_log, a.f.h0, a.dlast, a.hseg, a.gseg, a.sdt, chains, a.f.dim, a.f.dstate,
                a.nseg);
            err = cudaGetLastError();
        }
    }
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(scan_bwd_kernel<io_t, NPL, G, UA, kBwdFull, EX>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::kSmem));
    if (err == cudaSuccess) {
        scan_bwd_kernel<io_t, NPL, G, UA, kBwdFull, EX>
            <<<unsigned(ctas * nseg), C::NTH, C::kSmem, stream>>>(a, int(dblocks), vec_red);
        err = cudaGetLastError();
    }
    if (seg_mem) {
        const cudaError_t ferr = scratch_free(seg_mem, stream);
        if (err == cudaSuccess) err = ferr;
    }
    return err;
}

// The plain backward, or (h0, resets, dh0 or a final-state gradient given)
// the extended one.
template <typename io_t, int NPL, int G, int UA = 2>
cudaError_t launch_bwd(const BwdArgs& a, bool vec_red, cudaStream_t stream) {
    if (a.f.h0 || a.f.reset || a.dh0 || a.dlast)
        return launch_bwd_impl<io_t, NPL, G, UA, true>(a, vec_red, stream);
    return launch_bwd_impl<io_t, NPL, G, UA, false>(a, vec_red, stream);
}

// Tile by dstate: NPL states per lane, G lanes per chain (G * NPL >= N).
// Four states per lane up to dstate 64: more lanes per chain give more warps
// to hide latency, and measured faster on B300 than eight states per lane
// (Mamba-1.4B-style layer at dstate 16: 3.2 ms vs 4.3 ms with 8 x 2; 2 x 2048
// x 8192 at dstate 64: 6.1 vs 7.2 ms with 8 x 8; 4 x 2048 x 4096 at dstate
// 32: 2.8 vs 3.1 ms with 8 x 4).  The adjoint's step loop is unrolled by two,
// which keeps the 4-state tiles at 128 registers (8 CTAs per SM).
// MAMBA_BWD_TILE selects the 8-state tiles instead: 1 for dstate <= 16 (8 x 2),
// 3 for dstate 17..64 (8 x 4, 8 x 8).
template <typename io_t>
cudaError_t dispatch_bwd(const BwdArgs& a, bool vec_red, cudaStream_t stream) {
    const int N = a.f.dstate;
    const char* v = getenv("MAMBA_BWD_TILE");
    const int tile = v ? atoi(v) : 0;
    if (tile == 1 && N <= 16) return launch_bwd<io_t, 8, 2>(a, vec_red, stream);
    if (tile == 3 && N > 16 && N <= 32) return launch_bwd<io_t, 8, 4>(a, vec_red, stream);
    if (tile == 3 && N > 32 && N <= 64) return launch_bwd<io_t, 8, 8>(a, vec_red, stream);
    if (N <= 8) return launch_bwd<io_t, 4, 2>(a, vec_red, stream);
    if (N <= 16) return launch_bwd<io_t, 4, 4>(a, vec_red, stream);
    if (N <= 32) return launch_bwd<io_t, 4, 8>(a, vec_red, stream);
    if (N <= 64) return launch_bwd<io_t, 4, 16>(a, vec_red, stream);
    if (N <= 128) return launch_bwd<io_t, 8, 16>(a, vec_red, stream);
    return launch_bwd<io_t, 8, 32>(a, vec_red, stream);
}

}  // namespace

cudaError_t launch_scan_bwd(const ScanBwdArgs& s, bool bf16, cudaStream_t stream) {
    return launch_scan_bwd_ex(s, nullptr, bf16, stream);
}

cudaError_t launch_scan_bwd_ex(const ScanBwdArgs& s, float* dh0, bool bf16, cudaStream_t stream) {
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
    if (chains == 0 || nchunks == 0) {  // no steps: the final state is h0 itself
        const size_t nst = size_t(chains) * s.f.dstate * sizeof(float);
        if (dh0 && chains > 0)
            err = s.dlast ? cudaMemcpyAsync(dh0, s.dlast, nst, cudaMemcpyDeviceToDevice, stream)
                          : cudaMemsetAsync(dh0, 0, nst, stream);
        return err;
    }
    // checkpoints: the state at the start of every chunk, stream-ordered scratch
    void* ck = nullptr;
    const size_t ckb = size_t(chains) * nchunks * s.f.dstate * sizeof(float);
    if ((err = scratch_alloc(&ck, ckb, stream)) != cudaSuccess) return err;
    BwdArgs a;
    static_cast<ScanBwdArgs&>(a) = s;
    a.ckpt = static_cast<float*>(ck);
    a.dh0 = dh0;
    // 16-byte atomics on dB / dC need rows of whole float4 and aligned bases
    const bool vec_red = s.f.dstate % 4 == 0 && (reinterpret_cast<uintptr_t>(s.dB) & 15) == 0 &&
                         (reinterpret_cast<uintptr_t>(s.dC) & 15) == 0;
    err = bf16 ? dispatch_bwd<__nv_bfloat16>(a, vec_red, stream)
               : dispatch_bwd<float>(a, vec_red, stream);
    const cudaError_t ferr = scratch_free(ck, stream);
    return err != cudaSuccess ? err : ferr;
}

}  // namespace mamba
