// Fused selective-scan forward kernels for sm_103a.
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
//   A. B and C of the chunk are in shared memory (bulk copies issued ahead of
//      time) and are widened once to fp32.  Per element, dt = softplus(delta +
//      bias) and dt*u are computed once, two elements per packed f32x2
//      instruction, and left in shared memory for the state threads.
//   B. The recurrence, two states per packed f32x2 instruction: per step and
//      state one ex2 on the SFU, a multiply for dt*A, a multiply for dt*u*B,
//      an fma for h and an fma for the C contraction.  The operands and the
//      exponentials of step t+1 are issued before the state update of step t,
//      so the SFU and shared-memory latencies overlap the fma chain.  Each
//      thread leaves one partial sum of C.h per step in shared memory.
//   C. Per (chain, step): sum the G partials, add D*u, gate with SiLU(z),
//      round and store y.
//
// Two kernels share phases A to C and differ in how u, delta and z arrive:
//   scan_tma_kernel  -- 2-D tensor-map bulk copies (cp.async.bulk.tensor) of
//                       [CH chains x T steps] tiles into a ring of S stages,
//                       issued S-1 chunks ahead, so that enough bytes are in
//                       flight per SM to stream from HBM; out-of-range rows
//                       and the ragged time tail are zero-filled by the copy.
//                       Used whenever the rows are 16-byte aligned.
//   scan_reg_kernel  -- 128-bit (or element-wise) loads prefetched into
//                       registers one chunk ahead; the fallback for rows that
//                       are not 16-byte aligned.
#include <cuda.h>
#include <stdlib.h>

#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "scratch_pool.cuh"

namespace mamba {

// Error word of this kernel family (see mbar_wait).
__device__ unsigned int g_scan_error;

// Wait for a bulk copy into shared memory; a wait that gives up sets the
// error word and makes this thread's later waits short (see mbar_wait_n).
__device__ __forceinline__ void wait_copy(uint64_t* bar, uint32_t parity, bool& failed) {
    if (!mbar_wait_n(bar, parity, failed ? kWaitLimitAfterFailure : kWaitLimit)) {
        failed = true;
        atomicOr(&g_scan_error, kErrWaitTimeout);
    }
}

namespace {

__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2 splat2(float v) { return pack2(v, v); }

// Elements (2q, 2q+1) of a vector of io values packed in 32-bit words, widened
// to fp32.  fp32: word pair (2q, 2q+1).  bf16: word q holds both elements.
template <typename io_t, typename V>
__device__ __forceinline__ f32x2 get_pair(const V& v, int q) {
    const unsigned* w = reinterpret_cast<const unsigned*>(&v);
    if constexpr (sizeof(io_t) == 4) {
        return pack2(__uint_as_float(w[2 * q]), __uint_as_float(w[2 * q + 1]));
    } else {
        return pack2(__uint_as_float(w[q] << 16), __uint_as_float(w[q] & 0xffff0000u));
    }
}

// softplus of one value: the bf16 path uses the SFU formulation of
// softplus_fast, the fp32 path libdevice expf/log1pf.
template <typename io_t>
__device__ __forceinline__ float softplus_io(float x) {
    if constexpr (sizeof(io_t) == 4) {
        return softplus_accurate(x);
    } else {
        return softplus_fast(x);
    }
}

// The same on a pair (each lane exactly as softplus_io).
template <typename io_t>
__device__ __forceinline__ f32x2 softplus_pair(f32x2 x) {
    float x0, x1;
    unpack2(x, x0, x1);
    return pack2(softplus_io<io_t>(x0), softplus_io<io_t>(x1));
}

// y * SiLU(z) on a pair (each lane exactly as gate_silu).
__device__ __forceinline__ f32x2 gate_pair(f32x2 y, f32x2 z) {
    float y0, y1, z0, z1;
    unpack2(y, y0, y1);
    unpack2(z, z0, z1);
    return pack2(gate_silu(y0, z0), gate_silu(y1, z1));
}

// Element e of a vector of io values (bf16: the upper half-word is the odd one).
template <typename io_t, typename V>
__device__ __forceinline__ float io_elem(const V& v, int e) {
    const unsigned* w = reinterpret_cast<const unsigned*>(&v);
    if constexpr (sizeof(io_t) == 4) {
        return __uint_as_float(w[e]);
    } else {
        return __uint_as_float((e & 1) ? (w[e >> 1] & 0xffff0000u) : (w[e >> 1] << 16));
    }
}

// Pack NQ pairs of fp32 into io values (bf16: round to nearest even).
template <typename io_t, int NPAIR>
__device__ __forceinline__ void pack_out(const f32x2 (&val)[NPAIR], unsigned (&w)[NPAIR * sizeof(io_t) / 2]) {
#pragma unroll
    for (int q = 0; q < NPAIR; ++q) {
        float a, b;
        unpack2(val[q], a, b);
        if constexpr (sizeof(io_t) == 4) {
            w[2 * q] = __float_as_uint(a);
            w[2 * q + 1] = __float_as_uint(b);
        } else {
            const __nv_bfloat162 pr = __floats2bfloat162_rn(a, b);
            w[q] = *reinterpret_cast<const unsigned*>(&pr);
        }
    }
}

// Column of chain `cc` at step t in the (dt, dt*u) buffer: the XOR keeps the
// per-element writes of phase A and the per-step reads of phase B free of
// shared-memory bank conflicts.
template <int CH>
__device__ __forceinline__ int du_col(int t, int cc) {
    return cc ^ (((t >> 2) << 1) & (CH - 1));
}

// Partial sums of the recurrence live in a quad-major layout: 16-byte chunk
// (steps 4q..4q+3) of row `row` is chunk q * ROWS + (row ^ q).  The XOR keeps
// both the per-step writes (32 consecutive rows, one quad) and the
// per-element reads (G rows of 8 chains x 4 quads) free of bank conflicts.
template <int ROWS>
__device__ __forceinline__ int yunit(int q, int row) {
    static_assert(ROWS % 16 == 0, "rows come in groups of 16");
    return q * ROWS + (row ^ q);
}

// ---- phase B ------------------------------------------------------------
// The recurrence over one chunk for one thread: NQ quads of states of chain
// c (state group g).  sdu: (dt, dt, dt*u, dt*u) per [step][column]; sB, sC:
// fp32 [T][NP]; sy: partial sums [NTH rows][T], 16-byte chunks swizzled.
template <bool ACC, int NPL, int G, int CH, int T>
__device__ __forceinline__ void recurrence(const float4* sdu, const float* sB, const float* sC,
                                           float* sy, f32x2 (&h)[NPL / 2],
                                           const f32x2 (&A2)[NPL / 2], int c, int g, int tid,
                                           int tlen) {
    constexpr int NQ = NPL / 4, NP = NPL * G;
    const ulonglong2* du2 = reinterpret_cast<const ulonglong2*>(sdu);
    const ulonglong2* b2 = reinterpret_cast<const ulonglong2*>(sB) + g * NQ;
    const ulonglong2* c2 = reinterpret_cast<const ulonglong2*>(sC) + g * NQ;
    float4* y4 = reinterpret_cast<float4*>(sy);
    struct Step {
        ulonglong2 sd;  // (dt, dt), (dt*u, dt*u)
        f32x2 a[2 * NQ];
        ulonglong2 bq[NQ], cq[NQ];
    };
    auto fetch = [&](int t, Step& st) {
        st.sd = du2[t * CH + du_col<CH>(t, c)];
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            st.a[2 * q] = abar_exp2_pair<ACC>(mul2(st.sd.x, A2[2 * q]));
            st.a[2 * q + 1] = abar_exp2_pair<ACC>(mul2(st.sd.x, A2[2 * q + 1]));
            st.bq[q] = b2[t * (NP / 4) + q];
            st.cq[q] = c2[t * (NP / 4) + q];
        }
    };
    auto update = [&](const Step& st) -> float {
        // two accumulators halve the dependent chain of C.h within a step
        f32x2 acc0 = splat2(0.f), acc1 = splat2(0.f);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            h[2 * q] = fma2(st.a[2 * q], h[2 * q], mul2(st.sd.y, st.bq[q].x));
            h[2 * q + 1] = fma2(st.a[2 * q + 1], h[2 * q + 1], mul2(st.sd.y, st.bq[q].y));
            acc0 = fma2(st.cq[q].x, h[2 * q], acc0);
            acc1 = fma2(st.cq[q].y, h[2 * q + 1], acc1);
        }
        float lo, hi;
        unpack2(add2(acc0, acc1), lo, hi);
        return lo + hi;
    };
    Step cur;
    fetch(0, cur);
    if (tlen == T) {
#pragma unroll
        for (int tt = 0; tt < T; tt += 4) {
            float part[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                Step nxt;
                if (tt + j + 1 < T) fetch(tt + j + 1, nxt);
                part[j] = update(cur);
                if (tt + j + 1 < T) cur = nxt;
            }
            y4[yunit<CH * G>(tt / 4, tid)] = make_float4(part[0], part[1], part[2], part[3]);
        }
    } else {
        for (int tt = 0; tt < tlen; tt += 4) {
            float part[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int t = tt + j;
                Step nxt;
                if (t + 1 < tlen) fetch(t + 1, nxt);
                part[j] = t < tlen ? update(cur) : 0.f;
                if (t + 1 < tlen) cur = nxt;
            }
            y4[yunit<CH * G>(tt / 4, tid)] = make_float4(part[0], part[1], part[2], part[3]);
        }
    }
}

// Sum of the G partials of chain cc over the 4 steps [4*q4, 4*q4+4) of the
// chunk, as two pairs.
template <int G, int T, int ROWS>
__device__ __forceinline__ void partial_sums(const float* sy, int cc, int q4, f32x2& s01,
                                             f32x2& s23) {
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
        const int r = cc * G + gg;
        const ulonglong2 v = reinterpret_cast<const ulonglong2*>(sy)[yunit<ROWS>(q4, r)];
        s01 = gg == 0 ? v.x : add2(s01, v.x);
        s23 = gg == 0 ? v.y : add2(s23, v.y);
    }
}

// Widen the chunk's B and C (raw io values [T][N]) into fp32 [T][NP], with
// zero padding for states N..NP-1.
template <typename io_t, int NP, int T, int NTH>
__device__ __forceinline__ void widen_bc(const unsigned char* rawB, const unsigned char* rawC,
                                         float* sB, float* sC, int N, int tid) {
    constexpr int ES = sizeof(io_t);
    if (N == NP && (N * ES) % 16 == 0) {
        constexpr int PER = 16 / ES;  // io values per 16 bytes
        const uint4* rb = reinterpret_cast<const uint4*>(rawB);
        const uint4* rc = reinterpret_cast<const uint4*>(rawC);
        for (int it = tid; it < T * NP / PER; it += NTH) {
            const uint4 vb = rb[it], vc = rc[it];
            ulonglong2* ob = reinterpret_cast<ulonglong2*>(sB + it * PER);
            ulonglong2* oc = reinterpret_cast<ulonglong2*>(sC + it * PER);
#pragma unroll
            for (int q = 0; q < PER / 4; ++q) {
                ob[q] = make_ulonglong2(get_pair<io_t>(vb, 2 * q), get_pair<io_t>(vb, 2 * q + 1));
                oc[q] = make_ulonglong2(get_pair<io_t>(vc, 2 * q), get_pair<io_t>(vc, 2 * q + 1));
            }
        }
    } else {
        const io_t* rb = reinterpret_cast<const io_t*>(rawB);
        const io_t* rc = reinterpret_cast<const io_t*>(rawC);
        for (int idx = tid; idx < T * NP; idx += NTH) {
            const int t = idx / NP, n = idx % NP;
            const bool ok = n < N;
            sB[idx] = ok ? float(rb[t * N + n]) : 0.f;
            sC[idx] = ok ? float(rc[t * N + n]) : 0.f;
        }
    }
}

// widen_bc with 8-byte pieces, so that more threads share the work (the
// element warps of the warp-specialised kernel: T * NP / 4 pieces of 4 values).
template <typename io_t, int NP, int T, int NTH>
__device__ __forceinline__ void widen_bc_split(const unsigned char* rawB,
                                               const unsigned char* rawC, float* sB, float* sC,
                                               int N, int tid) {
    if constexpr (sizeof(io_t) == 2) {
        if (N == NP && (N * 2) % 16 == 0) {
            const uint2* rb = reinterpret_cast<const uint2*>(rawB);
            const uint2* rc = reinterpret_cast<const uint2*>(rawC);
            uint2 vb[(T * NP / 4 + NTH - 1) / NTH], vc[(T * NP / 4 + NTH - 1) / NTH];
#pragma unroll
            for (int r = 0; r < (T * NP / 4 + NTH - 1) / NTH; ++r) {
                const int it = tid + r * NTH;
                if (it < T * NP / 4) {
                    vb[r] = rb[it];
                    vc[r] = rc[it];
                }
            }
#pragma unroll
            for (int r = 0; r < (T * NP / 4 + NTH - 1) / NTH; ++r) {
                const int it = tid + r * NTH;
                if (it < T * NP / 4) {
                    reinterpret_cast<ulonglong2*>(sB)[it] = make_ulonglong2(
                        get_pair<io_t>(vb[r], 0), get_pair<io_t>(vb[r], 1));
                    reinterpret_cast<ulonglong2*>(sC)[it] = make_ulonglong2(
                        get_pair<io_t>(vc[r], 0), get_pair<io_t>(vc[r], 1));
                }
            }
            return;
        }
    }
    widen_bc<io_t, NP, T, NTH>(rawB, rawC, sB, sC, N, tid);
}

// A2 = min(A * log2 e, -kA2Max) so that Abar = 2^(dt * A2) and a step with
// dt = +inf (a document boundary, see reset_dt) gives Abar = 0 exactly.  The
// cap changes nothing for |A| >= 1e-30 (A_log >= -69); padded states get
// A2 = -kA2Max with B = C = 0, so they stay zero.
constexpr float kA2Max = 1e-30f;

// dt written to the exponent lanes of a step that starts a new document:
// 2^(+inf * A2) = 0 wipes the state, while dt * u keeps the real dt.
constexpr float kResetDt = __builtin_inff();

template <int NPL, int G>
__device__ __forceinline__ void init_state(const ScanArgs& p, int64_t d, bool chain_ok, int g,
                                           f32x2 (&A2)[NPL / 2], f32x2 (&h)[NPL / 2]) {
#pragma unroll
    for (int q = 0; q < NPL / 2; ++q) {
        float a[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int n = g * NPL + 2 * q + e;
            const float v = (chain_ok && n < p.dstate)
                                ? -expf(__ldg(p.A_log + d * p.dstate + n)) * kLog2e
                                : 0.f;
            a[e] = fminf(v, -kA2Max);
        }
        A2[q] = pack2(a[0], a[1]);
        h[q] = splat2(0.f);
    }
}

template <int NPL, int G>
__device__ __forceinline__ void store_state(const ScanArgs& p, int64_t chain, int g,
                                            const f32x2 (&h)[NPL / 2]) {
    float* out = p.last_state + chain * p.dstate;
#pragma unroll
    for (int q = 0; q < NPL / 2; ++q) {
        float v[2];
        unpack2(h[q], v[0], v[1]);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int n = g * NPL + 2 * q + e;
            if (n < p.dstate) out[n] = v[e];
        }
    }
}

// State of NPL states per thread from / to an fp32 [N] row (segmented scan).
template <int NPL, int G>
__device__ __forceinline__ void load_state(const float* src, int N, int g, f32x2 (&h)[NPL / 2]) {
#pragma unroll
    for (int q = 0; q < NPL / 2; ++q) {
        const int n = g * NPL + 2 * q;
        h[q] = pack2(n < N ? src[n] : 0.f, n + 1 < N ? src[n + 1] : 0.f);
    }
}
template <int NPL, int G>
__device__ __forceinline__ void write_state(float* dst, int N, int g, const f32x2 (&h)[NPL / 2]) {
#pragma unroll
    for (int q = 0; q < NPL / 2; ++q) {
        float v0, v1;
        unpack2(h[q], v0, v1);
        const int n = g * NPL + 2 * q;
        if (n < N) dst[n] = v0;
        if (n + 1 < N) dst[n + 1] = v1;
    }
}

// =========================================================================
// Tensor-map (TMA) path
// =========================================================================
constexpr int kTmaT = 16;      // steps per chunk
constexpr int kTmaStages = 4;  // ring depth: copies run 3 chunks ahead

template <typename io_t, int NPL, int G, int CH>
struct TmaCfg {
    static constexpr int T = kTmaT, S = kTmaStages;
    static constexpr int NTH = CH * G, NP = NPL * G, ES = sizeof(io_t);
    static constexpr int PV = 4;                  // elements per thread access
    static constexpr int SEGROW = T / PV;
    static constexpr int NSEG = CH * SEGROW;
    static constexpr int SPT = (NSEG + NTH - 1) / NTH;
    static constexpr size_t rnd(size_t x) { return (x + 127) / 128 * 128; }
    static constexpr size_t kTile = rnd(size_t(CH) * T * ES);   // u, delta or z tile
    static constexpr size_t kRaw = rnd(size_t(T) * NP * ES);    // B or C, raw
    static constexpr size_t kStage = 3 * kTile + 2 * kRaw;
    static constexpr size_t kRing = 128;
    static constexpr size_t kBf = kRing + S * kStage;
    static constexpr size_t kDu = kBf + 2 * size_t(T) * NP * 4;
    static constexpr size_t kY = kDu + size_t(T) * CH * 16;
    static constexpr size_t kSmem = kY + size_t(NTH) * T * 4;
    using quad_t = std::conditional_t<ES == 2, uint2, uint4>;  // PV io values
};

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

template <typename io_t, int NPL, int G, int CH>
__global__ void __launch_bounds__(CH* G)
    scan_tma_kernel(const ScanArgs p, const __grid_constant__ CUtensorMap tm_u,
                    const __grid_constant__ CUtensorMap tm_d,
                    const __grid_constant__ CUtensorMap tm_z, const int dblocks) {
    using C = TmaCfg<io_t, NPL, G, CH>;
    constexpr int T = C::T, S = C::S, NTH = C::NTH, NP = C::NP, PV = C::PV;
    using quad_t = typename C::quad_t;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    float* sB = reinterpret_cast<float*>(smem + C::kBf);
    float* sC = sB + T * NP;
    float4* sdu = reinterpret_cast<float4*>(smem + C::kDu);
    float* sy = reinterpret_cast<float*>(smem + C::kY);
    auto tile = [&](int s, int which) { return smem + C::kRing + s * C::kStage + which * C::kTile; };
    auto raw = [&](int s, int which) {
        return smem + C::kRing + s * C::kStage + 3 * C::kTile + which * C::kRaw;
    };

    const int64_t L = p.seqlen, dim = p.dim;
    const int N = p.dstate;
    const int b = blockIdx.x / dblocks;
    const int64_t d0 = int64_t(blockIdx.x % dblocks) * CH;
    const int tid = threadIdx.x;
    const int c = tid / G, g = tid % G;
    const int64_t d = d0 + c;
    const bool chain_ok = d < dim;
    const int64_t nchunks = (L + T - 1) / T;
    const int row0 = int(int64_t(b) * dim + d0);
    const bool has_z = p.z != nullptr;
    const io_t* Bg = static_cast<const io_t*>(p.B) + int64_t(b) * L * N;
    const io_t* Cg = static_cast<const io_t*>(p.C) + int64_t(b) * L * N;

    auto issue = [&](int64_t k) {  // one thread
        const int s = int(k % S);
        const int tl = L - k * T < T ? int(L - k * T) : T;
        const uint32_t bc_bytes = uint32_t(tl) * N * C::ES;
        const uint32_t tile_bytes = uint32_t(CH) * T * C::ES;
        mbar_arrive_expect_tx(&bar[s], (has_z ? 3 : 2) * tile_bytes + 2 * bc_bytes);
        tma_load_2d(tile(s, 0), &tm_u, int(k * T), row0, &bar[s]);
        tma_load_2d(tile(s, 1), &tm_d, int(k * T), row0, &bar[s]);
        if (has_z) tma_load_2d(tile(s, 2), &tm_z, int(k * T), row0, &bar[s]);
        bulk_g2s(raw(s, 0), Bg + k * T * N, bc_bytes, &bar[s]);
        bulk_g2s(raw(s, 1), Cg + k * T * N, bc_bytes, &bar[s]);
    };

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
        fence_proxy_async_smem();
        for (int64_t k = 0; k < S - 1 && k < nchunks; ++k) issue(k);
    }
    f32x2 A2[NPL / 2], h[NPL / 2];
    init_state<NPL, G>(p, d, chain_ok, g, A2, h);
    __syncthreads();

    bool copy_failed = false;
    io_t* yy = static_cast<io_t*>(p.y);
    for (int64_t k = 0; k < nchunks; ++k) {
        const int s = int(k % S);
        const int64_t t0 = k * T;
        const int tlen = L - t0 < T ? int(L - t0) : T;
        wait_copy(&bar[s], uint32_t(k / S) & 1u, copy_failed);

        // ---- phase A ----
        widen_bc<io_t, NP, T, NTH>(raw(s, 0), raw(s, 1), sB, sC, N, tid);
#pragma unroll
        for (int i = 0; i < C::SPT; ++i) {
            const int sidx = tid + i * NTH;
            if (sidx >= C::NSEG) break;
            const int seg = sidx % C::SEGROW, cc = sidx / C::SEGROW;
            const int64_t dd = d0 + cc;
            const bool live = dd < dim && seg * PV < tlen;
            const quad_t vd = reinterpret_cast<const quad_t*>(tile(s, 1))[cc * C::SEGROW + seg];
            const quad_t vu = reinterpret_cast<const quad_t*>(tile(s, 0))[cc * C::SEGROW + seg];
            const f32x2 bias2 = splat2((dd < dim && p.delta_bias) ? __ldg(p.delta_bias + dd) : 0.f);
#pragma unroll
            for (int q = 0; q < PV / 2; ++q) {
                f32x2 dt = add2(get_pair<io_t>(vd, q), bias2);
                if (p.softplus) dt = softplus_pair<io_t>(dt);
                const f32x2 du = mul2(dt, get_pair<io_t>(vu, q));
                float dt0, dt1, du0, du1;
                unpack2(dt, dt0, dt1);
                unpack2(du, du0, du1);
                if (!live) dt0 = dt1 = du0 = du1 = 0.f;
                const int t = seg * PV + 2 * q;
                sdu[t * CH + du_col<CH>(t, cc)] = make_float4(dt0, dt0, du0, du0);
                sdu[(t + 1) * CH + du_col<CH>(t + 1, cc)] = make_float4(dt1, dt1, du1, du1);
            }
        }
        __syncthreads();
        // The stage consumed one chunk ago is free: refill it S-1 chunks ahead.
        if (tid == 0 && k + S - 1 < nchunks) {
            fence_proxy_async_smem();
            issue(k + S - 1);
        }

        // ---- phase B ----
        recurrence<sizeof(io_t) == 4, NPL, G, CH, T>(sdu, sB, sC, sy, h, A2, c, g, tid, tlen);
        __syncthreads();

        // ---- phase C ----
#pragma unroll
        for (int i = 0; i < C::SPT; ++i) {
            const int sidx = tid + i * NTH;
            if (sidx >= C::NSEG) break;
            const int seg = sidx % C::SEGROW, cc = sidx / C::SEGROW;
            const int64_t dd = d0 + cc;
            if (dd >= dim || seg * PV >= tlen) continue;
            f32x2 v[2];
            partial_sums<G, T, CH * G>(sy, cc, seg, v[0], v[1]);
            const quad_t vu = reinterpret_cast<const quad_t*>(tile(s, 0))[cc * C::SEGROW + seg];
            const f32x2 D2 = splat2(p.D ? __ldg(p.D + dd) : 0.f);
            v[0] = fma2(D2, get_pair<io_t>(vu, 0), v[0]);
            v[1] = fma2(D2, get_pair<io_t>(vu, 1), v[1]);
            if (has_z) {
                const quad_t vz = reinterpret_cast<const quad_t*>(tile(s, 2))[cc * C::SEGROW + seg];
                v[0] = gate_pair(v[0], get_pair<io_t>(vz, 0));
                v[1] = gate_pair(v[1], get_pair<io_t>(vz, 1));
            }
            unsigned w[PV * C::ES / 4];
            pack_out<io_t, 2>(v, w);
            *reinterpret_cast<quad_t*>(yy + (int64_t(b) * dim + dd) * L + t0 + seg * PV) =
                *reinterpret_cast<const quad_t*>(w);
        }
    }
    if (chain_ok && p.last_state) store_state<NPL, G>(p, int64_t(b) * dim + d, g, h);
}

// =========================================================================
// Warp-specialised tensor-map path
// =========================================================================
// Measured per 16-step chunk of the single-chain tile, two thirds of the
// time went to the per-element work (dt, dt*u before the recurrence; the
// G-partial sum, skip and gate after it) and to issuing and waiting for the
// bulk copies, all done by the same warps between barriers while the
// recurrence waited.  Here the CTA has two roles that overlap:
//   recurrence warps (NR threads) -- the state update of chunk k;
//   element warps (NE threads)    -- the bulk copies, the per-element
//                                    prologue of chunk k+1 (and the fp32
//                                    widening of its B and C) and the
//                                    epilogue of chunk k-1.
// Hand-off buffers are double-buffered and signalled with named barriers:
// "prologue of chunk k ready" (element warps arrive, recurrence warps wait)
// and "recurrence of chunk k done" (the reverse).
//
// A recurrence thread owns NPL states of P chains.  B and C of a step are
// shared by every channel of a batch row, so with P = 2 each B/C value read
// from shared memory serves two chains: per state update the thread reads
// 8/P bytes of B and C plus 16/NPL bytes of (dt, dt*u).
template <typename io_t, int P, int NPL, int G, int NR, int NE>
struct WsCfg {
    static constexpr int T = 16, S = 4;
    static constexpr int NTH = NR + NE;
    static constexpr int NGRP = NR / G;     // chain slots per chain set
    static constexpr int CH = P * NGRP;     // chains per CTA
    static constexpr int NP = NPL * G, ES = sizeof(io_t), PV = 4;
    static constexpr int SEGROW = T / PV;
    static constexpr int NSEG = CH * SEGROW;
    static constexpr int SPT = NSEG / NE;   // segments per element thread
    static constexpr int EW = NE / 32;         // element warps
    static constexpr int CW = CH / EW;         // chains per element warp
    static constexpr size_t rnd(size_t x) { return (x + 127) / 128 * 128; }
    static constexpr size_t kTile = rnd(size_t(CH) * T * ES);
    static constexpr size_t kRaw = rnd(size_t(T) * NP * ES);
    static constexpr size_t kStage = 3 * kTile + 2 * kRaw;
    static constexpr size_t kRing = 128;
    static constexpr size_t kBcBuf = 2 * size_t(T) * NP * 4;  // fp32 B and C
    static constexpr size_t kBc = kRing + S * kStage;
    static constexpr size_t kDuBuf = size_t(T) * CH * 16;
    static constexpr size_t kDu = kBc + 2 * kBcBuf;
    static constexpr size_t kYBuf = size_t(CH) * G * T * 4;
    static constexpr size_t kY = kDu + 2 * kDuBuf;
    static constexpr size_t kSmem = kY + 2 * kYBuf;
    using quad_t = std::conditional_t<ES == 2, uint2, uint4>;
    static_assert(NR % 32 == 0 && NE % 32 == 0, "roles are whole warps");
    static_assert(NSEG % NE == 0, "element threads share the segments evenly");
    static_assert(NE == 32 || NE == 64,
                  "one element warp copies B and C, or two: one copies B, the other C");
    static_assert(CW * SEGROW == 32 * SPT, "an element warp covers its chains exactly");
    static_assert((T * NP * ES) % (32 * 16) == 0, "B and C split into 16-byte pieces per lane");
    static_assert((size_t(CW) * T * ES) % 128 == 0, "per-warp tile rows stay 128-byte aligned");
    static_assert((CH & (CH - 1)) == 0, "chain count per CTA is a power of two");
};

// The recurrence over one chunk for P chains x NPL states of one thread (the
// multi-chain form of recurrence() above; rows of sy are chain * G + g).
template <bool ACC, int P, int NPL, int G, int CH, int T>
__device__ __forceinline__ void recurrence_multi(const float4* sdu, const float* sB,
                                                 const float* sC, float* sy,
                                                 f32x2 (&h)[P][NPL / 2],
                                                 const f32x2 (&A2)[P][NPL / 2],
                                                 const int (&cc)[P], int g, int tlen) {
    constexpr int NQ = NPL / 4, NP = NPL * G;
    const ulonglong2* du2 = reinterpret_cast<const ulonglong2*>(sdu);
    const ulonglong2* b2 = reinterpret_cast<const ulonglong2*>(sB) + g * NQ;
    const ulonglong2* c2 = reinterpret_cast<const ulonglong2*>(sC) + g * NQ;
    float4* y4 = reinterpret_cast<float4*>(sy);
    int row[P];
#pragma unroll
    for (int p = 0; p < P; ++p) row[p] = cc[p] * G + g;
    struct Step {
        ulonglong2 sd[P];  // (dt, dt), (dt*u, dt*u) per chain
        f32x2 a[P][2 * NQ];
        ulonglong2 bq[NQ], cq[NQ];
    };
    auto fetch = [&](int t, Step& st) {
#pragma unroll
        for (int p = 0; p < P; ++p) st.sd[p] = du2[t * CH + du_col<CH>(t, cc[p])];
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            st.bq[q] = b2[t * (NP / 4) + q];
            st.cq[q] = c2[t * (NP / 4) + q];
        }
#pragma unroll
        for (int p = 0; p < P; ++p) {
#pragma unroll
            for (int q = 0; q < 2 * NQ; ++q) st.a[p][q] = abar_exp2_pair<ACC>(mul2(st.sd[p].x, A2[p][q]));
        }
    };
    auto update = [&](const Step& st, float (&out)[P]) {
#pragma unroll
        for (int p = 0; p < P; ++p) {
            f32x2 acc = splat2(0.f);
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                h[p][2 * q] = fma2(st.a[p][2 * q], h[p][2 * q], mul2(st.sd[p].y, st.bq[q].x));
                h[p][2 * q + 1] =
                    fma2(st.a[p][2 * q + 1], h[p][2 * q + 1], mul2(st.sd[p].y, st.bq[q].y));
                acc = fma2(st.cq[q].x, h[p][2 * q], acc);
                acc = fma2(st.cq[q].y, h[p][2 * q + 1], acc);
            }
            float lo, hi;
            unpack2(acc, lo, hi);
            out[p] = lo + hi;
        }
    };
    Step cur;
    fetch(0, cur);
    if (tlen == T) {
#pragma unroll
        for (int tt = 0; tt < T; tt += 4) {
            float part[4][P];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                Step nxt;
                if (tt + j + 1 < T) fetch(tt + j + 1, nxt);
                update(cur, part[j]);
                if (tt + j + 1 < T) cur = nxt;
            }
#pragma unroll
            for (int p = 0; p < P; ++p)
                y4[yunit<CH * G>(tt / 4, row[p])] =
                    make_float4(part[0][p], part[1][p], part[2][p], part[3][p]);
        }
    } else {
        for (int tt = 0; tt < tlen; tt += 4) {
            float part[4][P];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int t = tt + j;
                Step nxt;
                if (t + 1 < tlen) fetch(t + 1, nxt);
                if (t < tlen) {
                    update(cur, part[j]);
                } else {
#pragma unroll
                    for (int p = 0; p < P; ++p) part[j][p] = 0.f;
                }
                if (t + 1 < tlen) cur = nxt;
            }
#pragma unroll
            for (int p = 0; p < P; ++p)
                y4[yunit<CH * G>(tt / 4, row[p])] =
                    make_float4(part[0][p], part[1][p], part[2][p], part[3][p]);
        }
    }
}

// State-only recurrence over one chunk (no C, no partial sums): the summary
// pass of a segmented scan needs only the state at the end of the segment.
template <bool ACC, int NPL, int G, int CH, int T>
__device__ __forceinline__ void recurrence_state(const float4* sdu, const float* sB,
                                                 f32x2 (&h)[NPL / 2], const f32x2 (&A2)[NPL / 2],
                                                 int c, int g, int tlen) {
    constexpr int NQ = NPL / 4, NP = NPL * G;
    const ulonglong2* du2 = reinterpret_cast<const ulonglong2*>(sdu);
    const ulonglong2* b2 = reinterpret_cast<const ulonglong2*>(sB) + g * NQ;
    struct Step {
        ulonglong2 sd;
        f32x2 a[2 * NQ];
        ulonglong2 bq[NQ];
    };
    auto fetch = [&](int t, Step& st) {
        st.sd = du2[t * CH + du_col<CH>(t, c)];
#pragma unroll
        for (int q = 0; q < NQ; ++q) st.bq[q] = b2[t * (NP / 4) + q];
#pragma unroll
        for (int q = 0; q < 2 * NQ; ++q) st.a[q] = abar_exp2_pair<ACC>(mul2(st.sd.x, A2[q]));
    };
    auto update = [&](const Step& st) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            h[2 * q] = fma2(st.a[2 * q], h[2 * q], mul2(st.sd.y, st.bq[q].x));
            h[2 * q + 1] = fma2(st.a[2 * q + 1], h[2 * q + 1], mul2(st.sd.y, st.bq[q].y));
        }
    };
    Step cur;
    fetch(0, cur);
    if (tlen == T) {
#pragma unroll
        for (int t = 0; t < T; ++t) {
            Step nxt;
            if (t + 1 < T) fetch(t + 1, nxt);
            update(cur);
            if (t + 1 < T) cur = nxt;
        }
    } else {
        for (int t = 0; t < tlen; ++t) {
            Step nxt;
            if (t + 1 < tlen) fetch(t + 1, nxt);
            update(cur);
            if (t + 1 < tlen) cur = nxt;
        }
    }
}

__device__ __forceinline__ void named_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_arrive(int id, int count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}
constexpr int kBarReady = 1;  // + (chunk & 1): prologue of the chunk written
constexpr int kBarDone = 3;   // + (chunk & 1): recurrence of the chunk done

// MODE kScanFull: the scan of a whole sequence (sg.nseg == 1) or, in a
//   segmented scan, of segment s of every chain, starting from the state that
//   the carry pass left in sg.hcarry.
// MODE kScanSummary: segment s < nseg - 1 of a segmented scan from a zero
//   state, writing only the state at its end and the sum of its dt (no y).
constexpr int kScanFull = 0, kScanSummary = 1;

// FAST: the gate z is given, softplus is on and there is no reset mask (the
// common case, compiled without those run-time tests and without the
// per-element reset decoding; h0 and a split's carried state are read once
// per CTA either way).
template <typename io_t, int P, int NPL, int G, int NR, int NE, int MINB, int MODE,
          bool FAST = false>
__global__ void __launch_bounds__(NR + NE, MINB)
    scan_ws_kernel(const ScanArgs p, const __grid_constant__ CUtensorMap tm_u,
                   const __grid_constant__ CUtensorMap tm_d,
                   const __grid_constant__ CUtensorMap tm_z, const int dblocks,
                   const SegArgs sg) {
    using C = WsCfg<io_t, P, NPL, G, NR, NE>;
    static_assert(MODE == kScanFull || P == 1, "the summary pass uses one chain per thread");
    constexpr int T = C::T, S = C::S, NTH = C::NTH, NP = C::NP, PV = C::PV, CH = C::CH;
    constexpr int SPT = C::SPT;
    using quad_t = typename C::quad_t;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    auto stage = [&](int k) { return smem + C::kRing + (k & (S - 1)) * C::kStage; };
    auto tile = [&](int k, int which) { return stage(k) + which * C::kTile; };
    auto raw = [&](int k, int which) { return stage(k) + 3 * C::kTile + which * C::kRaw; };
    auto bcbuf = [&](int k) { return reinterpret_cast<float*>(smem + C::kBc + (k & 1) * C::kBcBuf); };
    auto dubuf = [&](int k) { return reinterpret_cast<float4*>(smem + C::kDu + (k & 1) * C::kDuBuf); };
    auto ybuf = [&](int k) { return reinterpret_cast<float*>(smem + C::kY + (k & 1) * C::kYBuf); };

    const int L = int(p.seqlen);
    const int64_t dim = p.dim;
    const int N = p.dstate;
    // blockIdx.x = (b * dblocks + channel block) * grid_nseg + time segment
    const int tseg = blockIdx.x % sg.grid_nseg;
    const int cblk = blockIdx.x / sg.grid_nseg;
    const int b = cblk / dblocks;
    const int64_t d0 = int64_t(cblk % dblocks) * CH;
    const int t0 = tseg * sg.seg_len;
    const int Ls = L - t0 < sg.seg_len ? L - t0 : sg.seg_len;  // steps of this segment
    const int tid = threadIdx.x;
    const int nchunks = (Ls + T - 1) / T;
    const int row0 = int(int64_t(b) * dim + d0);
    const bool has_z = MODE == kScanFull && (FAST || p.z != nullptr);
    const io_t* Bg = static_cast<const io_t*>(p.B) + (int64_t(b) * L + t0) * N;
    const io_t* Cg = static_cast<const io_t*>(p.C) + (int64_t(b) * L + t0) * N;
    auto chunk_len = [&](int k) { return Ls - k * T < T ? Ls - k * T : T; };
    const int nc = sg.nseg - 1;  // carried states per chain

    // Each element warp w owns chains [w * CW, (w + 1) * CW) of the CTA and
    // copies its own rows of the u / delta / z tiles; warp 0 also copies B and
    // warp 1 C.  Every warp thus waits on its own mbarrier per stage and
    // refills a stage as soon as it has finished with it, with no barrier
    // across the element warps.
    constexpr int CW = C::CW;
    auto issue = [&](int k, int w) {  // lane 0 of element warp w
        const uint32_t bc_bytes = uint32_t(chunk_len(k)) * N * C::ES;
        const uint32_t rows_bytes = uint32_t(CW) * T * C::ES;
        uint64_t* br = &bar[(k & (S - 1)) * 2 + w];
        unsigned char* st = stage(k) + w * rows_bytes;
        mbar_arrive_expect_tx(br, (has_z ? 3 : 2) * rows_bytes + (3 - C::EW) * bc_bytes);
        tma_load_2d(st, &tm_u, t0 + k * T, row0 + w * CW, br);
        tma_load_2d(st + C::kTile, &tm_d, t0 + k * T, row0 + w * CW, br);
        if (has_z) tma_load_2d(st + 2 * C::kTile, &tm_z, t0 + k * T, row0 + w * CW, br);
        if (C::EW == 1) {
            bulk_g2s(raw(k, 0), Bg + int64_t(k) * T * N, bc_bytes, br);
            bulk_g2s(raw(k, 1), Cg + int64_t(k) * T * N, bc_bytes, br);
        } else {
            bulk_g2s(raw(k, w), (w == 0 ? Bg : Cg) + int64_t(k) * T * N, bc_bytes, br);
        }
    };

    if (tid == NR) {
        for (int s = 0; s < 2 * S; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncthreads();

    if (tid < NR) {
        // ---------------- recurrence warps ----------------
        const int grp = tid / G, g = tid % G;
        int cc[P];
        f32x2 A2[P][NPL / 2], h[P][NPL / 2];
#pragma unroll
        for (int q = 0; q < P; ++q) {
            cc[q] = grp + q * C::NGRP;
            init_state<NPL, G>(p, d0 + cc[q], d0 + cc[q] < dim, g, A2[q], h[q]);
            if (MODE == kScanFull && d0 + cc[q] < dim) {
                const int64_t chain = int64_t(b) * dim + d0 + cc[q];
                if (sg.hcarry)  // split: the carry pass left the entering state in slot tseg
                    load_state<NPL, G>(sg.hcarry + (chain * sg.nseg + tseg) * N, N, g, h[q]);
                else if (p.h0)
                    load_state<NPL, G>(p.h0 + chain * N, N, g, h[q]);
            }
        }
        for (int k = 0; k < nchunks; ++k) {
            named_sync(kBarReady + (k & 1), NTH);
            const float* sB = bcbuf(k);
            if constexpr (MODE == kScanSummary) {
                recurrence_state<sizeof(io_t) == 4, NPL, G, CH, T>(dubuf(k), sB, h[0], A2[0], cc[0], g, chunk_len(k));
            } else if constexpr (P == 1) {
                recurrence<sizeof(io_t) == 4, NPL, G, CH, T>(dubuf(k), sB, sB + T * NP, ybuf(k), h[0], A2[0], cc[0],
                                          g, tid, chunk_len(k));
            } else {
                recurrence_multi<sizeof(io_t) == 4, P, NPL, G, CH, T>(dubuf(k), sB, sB + T * NP, ybuf(k), h, A2, cc,
                                                   g, chunk_len(k));
            }
            named_arrive(kBarDone + (k & 1), NTH);
        }
#pragma unroll
        for (int q = 0; q < P; ++q) {
            if (d0 + cc[q] >= dim) continue;
            const int64_t chain = int64_t(b) * dim + d0 + cc[q];
            if (MODE == kScanSummary)  // end state of segment tseg from zero -> slot tseg + 1
                write_state<NPL, G>(sg.hcarry + (chain * sg.nseg + tseg + 1) * N, N, g, h[q]);
            else if (p.last_state && tseg == sg.nseg - 1)
                store_state<NPL, G>(p, chain, g, h[q]);
        }
        return;
    }

    // ---------------- element warps ----------------
    // Lane l of element warp w handles segment (l % SEGROW) of the chains
    // w * CW + l / SEGROW + i * (32 / SEGROW), i < SPT.  Their bias and D, and
    // every shared-memory offset the thread uses, are fixed for the whole
    // sequence.  One pass per chunk k finishes chunk k - 1 (partial sums, skip
    // term, gate, store of y) and prepares chunk k + 1 (dt, dt * u, fp32 B or
    // C), loading all of its shared-memory inputs first so that the two
    // halves' dependency chains overlap.
    const int te = tid - NR, w = te / 32, lane = te % 32;
    const int seg = lane % C::SEGROW;
    constexpr int ROWS = CH * G;
    int ec[SPT], tq[SPT], dub[SPT], yu[SPT][G];
    float bias[SPT], Dd[SPT];
    bool chain_ok[SPT];
    io_t* yg[SPT];
#pragma unroll
    for (int i = 0; i < SPT; ++i) {
        ec[i] = w * CW + lane / C::SEGROW + i * (32 / C::SEGROW);
        const int64_t dd = d0 + ec[i];
        chain_ok[i] = dd < dim;
        bias[i] = (chain_ok[i] && p.delta_bias) ? __ldg(p.delta_bias + dd) : 0.f;
        Dd[i] = (chain_ok[i] && p.D) ? __ldg(p.D + dd) : 0.f;
        tq[i] = ec[i] * C::SEGROW + seg;
        dub[i] = seg * PV * CH + (ec[i] ^ ((2 * seg) & (CH - 1)));  // du_col of steps 4*seg..+3
#pragma unroll
        for (int gg = 0; gg < G; ++gg) yu[i][gg] = yunit<ROWS>(seg, ec[i] * G + gg);
        yg[i] = static_cast<io_t*>(p.y) + (int64_t(b) * dim + dd) * L + t0 + seg * PV;
    }
    const bool all_chains = d0 + CH <= dim;
    if (lane == 0) {
        fence_proxy_async_smem();
        for (int k = 0; k < S && k < nchunks; ++k) issue(k, w);
    }
    __syncwarp();

    bool copy_failed = false;
    float dtsum[SPT];  // summary pass: sum of dt over the segment
#pragma unroll
    for (int i = 0; i < SPT; ++i) dtsum[i] = 0.f;
    // ke: chunk to finish (or -1), kp: chunk to prepare (or -1)
    auto pass = [&](int ke, int kp) {
        if (MODE == kScanSummary) ke = -1;
        // ---- loads ----
        ulonglong2 ps[SPT][G];
        quad_t eu[SPT], ez[SPT], pd[SPT], pu[SPT];
        if (ke >= 0) {
            const ulonglong2* sy = reinterpret_cast<const ulonglong2*>(ybuf(ke));
            const quad_t* tu = reinterpret_cast<const quad_t*>(tile(ke, 0));
            const quad_t* tz = reinterpret_cast<const quad_t*>(tile(ke, 2));
#pragma unroll
            for (int i = 0; i < SPT; ++i) {
#pragma unroll
                for (int gg = 0; gg < G; ++gg) ps[i][gg] = sy[yu[i][gg]];
                eu[i] = tu[tq[i]];
                if (has_z) ez[i] = tz[tq[i]];
            }
        }
        constexpr int BCV = T * NP * C::ES / 32 / 16;  // 16-byte pieces of B or C per lane
        constexpr int NBC = 3 - C::EW;                 // B and C, or the warp's one of them
        uint4 rbc[NBC][BCV];
        // document boundaries of this lane's PV steps: one byte each (4-byte
        // aligned: the row length and every offset are multiples of 4)
        uint32_t rsw = 0;
        if (!FAST && kp >= 0 && p.reset && seg * PV < chunk_len(kp))
            rsw = __ldg(reinterpret_cast<const uint32_t*>(p.reset + int64_t(b) * L + t0 +
                                                          kp * T + seg * PV));
        if (kp >= 0) {
            wait_copy(&bar[(kp & (S - 1)) * 2 + w], uint32_t(kp / S) & 1u, copy_failed);
            const quad_t* td = reinterpret_cast<const quad_t*>(tile(kp, 1));
            const quad_t* tu = reinterpret_cast<const quad_t*>(tile(kp, 0));
#pragma unroll
            for (int i = 0; i < SPT; ++i) {
                pd[i] = td[tq[i]];
                pu[i] = tu[tq[i]];
            }
#pragma unroll
            for (int x = 0; x < NBC; ++x) {
                const uint4* rw = reinterpret_cast<const uint4*>(raw(kp, NBC == 2 ? x : w));
#pragma unroll
                for (int r = 0; r < BCV; ++r) rbc[x][r] = rw[lane * BCV + r];
            }
        }
        // ---- finish chunk ke ----
        if (ke >= 0) {
            const bool seg_live = seg * PV < chunk_len(ke);
#pragma unroll
            for (int i = 0; i < SPT; ++i) {
                // scalar fp32 throughout: every value here passes through the
                // SFU, so packed pairs would only add register moves
                float v[PV];
#pragma unroll
                for (int e = 0; e < PV; ++e) {
                    float acc = reinterpret_cast<const float*>(&ps[i][0])[e];
#pragma unroll
                    for (int gg = 1; gg < G; ++gg)
                        acc = __fadd_rn(acc, reinterpret_cast<const float*>(&ps[i][gg])[e]);
                    acc = __fmaf_rn(Dd[i], io_elem<io_t>(eu[i], e), acc);
                    v[e] = has_z ? gate_silu(acc, io_elem<io_t>(ez[i], e)) : acc;
                }
                f32x2 vp[2] = {pack2(v[0], v[1]), pack2(v[2], v[3])};
                unsigned wd[PV * C::ES / 4];
                pack_out<io_t, 2>(vp, wd);
                if (chain_ok[i] && seg_live)
                    *reinterpret_cast<quad_t*>(yg[i] + int64_t(ke) * T) =
                        *reinterpret_cast<const quad_t*>(wd);
            }
        }
        // ---- prepare chunk kp ----
        if (kp >= 0) {
            float4 o[SPT][PV];
#pragma unroll
            for (int i = 0; i < SPT; ++i) {
#pragma unroll
                for (int e = 0; e < PV; ++e) {
                    float dt = __fadd_rn(io_elem<io_t>(pd[i], e), bias[i]);
                    if (FAST || p.softplus) dt = softplus_io<io_t>(dt);
                    const float du = __fmul_rn(dt, io_elem<io_t>(pu[i], e));
                    // exponent lanes of a step that starts a document: +inf
                    const float de = ((rsw >> (8 * e)) & 0xffu) ? kResetDt : dt;
                    o[i][e] = make_float4(de, de, du, du);
                }
            }
            if (!all_chains || chunk_len(kp) < T) {  // zero steps past the end, dead chains
                const int tl = chunk_len(kp);
#pragma unroll
                for (int i = 0; i < SPT; ++i)
#pragma unroll
                    for (int e = 0; e < PV; ++e)
                        if (!chain_ok[i] || seg * PV + e >= tl) o[i][e] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (MODE == kScanSummary) {
#pragma unroll
                for (int i = 0; i < SPT; ++i)
#pragma unroll
                    for (int e = 0; e < PV; ++e) dtsum[i] += o[i][e].x;
            }
            float4* sdu = dubuf(kp);
#pragma unroll
            for (int i = 0; i < SPT; ++i)
#pragma unroll
                for (int e = 0; e < PV; ++e) sdu[dub[i] + e * CH] = o[i][e];
            // fp32 copy of B and C (one element warp), or of this warp's B
            // (w = 0) or C (w = 1)
#pragma unroll
            for (int x = 0; x < NBC; ++x) {
                float* dst = bcbuf(kp) + (NBC == 2 ? x : w) * T * NP + lane * BCV * (16 / C::ES);
#pragma unroll
                for (int r = 0; r < BCV; ++r) {
                    if constexpr (C::ES == 2) {
                        reinterpret_cast<ulonglong2*>(dst)[2 * r] = make_ulonglong2(
                            get_pair<io_t>(rbc[x][r], 0), get_pair<io_t>(rbc[x][r], 1));
                        reinterpret_cast<ulonglong2*>(dst)[2 * r + 1] = make_ulonglong2(
                            get_pair<io_t>(rbc[x][r], 2), get_pair<io_t>(rbc[x][r], 3));
                    } else {
                        reinterpret_cast<uint4*>(dst)[r] = rbc[x][r];
                    }
                }
            }
        }
    };

    if (nchunks == 0) return;  // (a segment is never empty; only a whole empty sequence)
    pass(-1, 0);
    named_arrive(kBarReady + 0, NTH);
    if (nchunks > 1) {
        pass(-1, 1);
        named_arrive(kBarReady + 1, NTH);
    }
    for (int j = 1; j <= nchunks; ++j) {
        named_sync(kBarDone + ((j - 1) & 1), NTH);
        const int kp = j + 1 < nchunks ? j + 1 : -1;
        pass(j - 1, kp);
        if (kp >= 0) named_arrive(kBarReady + (kp & 1), NTH);
        // this warp no longer reads the stage of chunk j - 1: refill it
        __syncwarp();
        if (lane == 0 && j - 1 + S < nchunks) {
            fence_proxy_async_smem();
            issue(j - 1 + S, w);
        }
    }
    if (MODE == kScanSummary) {
        // the SEGROW lanes of a chain hold its dt sums over disjoint steps
#pragma unroll
        for (int i = 0; i < SPT; ++i) {
#pragma unroll
            for (int off = 1; off < C::SEGROW; off *= 2)
                dtsum[i] += __shfl_xor_sync(0xffffffffu, dtsum[i], off);
            if (seg == 0 && chain_ok[i])
                sg.sdt[(int64_t(b) * dim + d0 + ec[i]) * nc + tseg] = dtsum[i];
        }
    }
}

// =========================================================================
// Paired-chain tensor-map path (dstate == 4*G exactly)
// =========================================================================
// Two observations shape this kernel.
//  * Shared-memory bandwidth: a 128-bit shared load costs four wavefronts per
//    warp even when every lane reads the same address, so delivering B and C
//    to each chain separately costs 8 bytes per state update.  Here each
//    thread owns 4 states (n = 4g..4g+3) of TWO adjacent chains: one load of
//    B and C (raw io values, widened in registers) serves both, and (dt,
//    dt*u) of both chains arrive in one 16-byte load.  dt*A is paired across
//    the two chains, B*dt*u and the state across the 4 states of one chain.
//  * Latency: each chain is a serial walk over the whole sequence, so the
//    time one warp needs per step bounds the kernel when the batch is small.
//    The operands and exponentials of step t+1 are issued before the update
//    of step t, and the per-element work of the neighbouring chunks (dt and
//    dt*u of chunk k+1, the epilogue of chunk k-1) is interleaved with the
//    recurrence of chunk k, four steps at a time; one CTA barrier per chunk,
//    (dt, dt*u) and the partial sums are double-buffered.
template <typename io_t, int G>
struct PairCfg {
    static constexpr int N = 4 * G, ES = sizeof(io_t), PV = 4, NPL = 4;
    // Large B/C stages (fp32, dstate 64 and up) would leave too few CTAs per
    // SM with double buffers: there the per-element phases run between two
    // barriers instead of being interleaved with the recurrence.
    static constexpr bool IL = N * ES < 256;
    static constexpr int NBUF = IL ? 2 : 1;
    static constexpr int T = 16;                     // steps per chunk
    static constexpr int S = N * ES >= 128 || G == 1 ? 4 : 8;  // ring depth (power of two)
    static constexpr int NGRP = T / 4;          // 4-step groups per chunk
    static constexpr int NTH = 64;
    static constexpr int NPAIR = NTH / G;  // chain pairs per CTA
    static constexpr int CH = 2 * NPAIR;   // chains per CTA
    static constexpr int SEGROW = T / PV;
    static constexpr int NSEG = CH * SEGROW;
    static constexpr int SPT = (NSEG + NTH - 1) / NTH;
    static constexpr size_t rnd(size_t x) { return (x + 127) / 128 * 128; }
    static constexpr size_t kTile = rnd(size_t(CH) * T * ES);
    static constexpr size_t kRaw = rnd(size_t(T) * N * ES);
    static constexpr size_t kStage = 3 * kTile + 2 * kRaw;
    static constexpr size_t kRing = 128;
    static constexpr size_t kSdBuf = size_t(T) * NPAIR * 16;      // [T][NPAIR] float4
    static constexpr size_t kSd = kRing + S * kStage;
    static constexpr size_t kYBuf = size_t(CH) * G * T * 4;       // [CH*G rows][T]
    static constexpr size_t kY = kSd + NBUF * kSdBuf;
    static constexpr size_t kSmem = kY + NBUF * kYBuf;
    using quad_t = std::conditional_t<ES == 2, uint2, uint4>;
    static_assert(CH <= 256, "tensor-map box height");
    static_assert((S & (S - 1)) == 0, "ring depth must be a power of two");
};

// Column of chain pair p at step t in the (dt, dt*u) buffer.
template <int NPAIR>
__device__ __forceinline__ int pair_col(int t, int p) {
    return p ^ ((t >> 2) & (NPAIR - 1));
}

template <typename io_t, int G>
__global__ void __launch_bounds__(64)
    scan_pair_kernel(const ScanArgs p, const __grid_constant__ CUtensorMap tm_u,
                     const __grid_constant__ CUtensorMap tm_d,
                     const __grid_constant__ CUtensorMap tm_z, const int dblocks) {
    using C = PairCfg<io_t, G>;
    constexpr int T = C::T, S = C::S, NTH = C::NTH, NPAIR = C::NPAIR, CH = C::CH, N = C::N;
    constexpr int PV = C::PV, NGRP = C::NGRP, SPT = C::SPT;
    using quad_t = typename C::quad_t;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    // chunk indices fit in 32 bits (seqlen < 2^31 on this path)
    auto stage = [&](int k) { return smem + C::kRing + (k & (S - 1)) * C::kStage; };
    auto tile = [&](int k, int which) { return stage(k) + which * C::kTile; };
    auto raw = [&](int k, int which) { return stage(k) + 3 * C::kTile + which * C::kRaw; };
    auto sdbuf = [&](int k) {
        return reinterpret_cast<float*>(smem + C::kSd + (k & (C::NBUF - 1)) * C::kSdBuf);
    };
    auto ybuf = [&](int k) {
        return reinterpret_cast<float*>(smem + C::kY + (k & (C::NBUF - 1)) * C::kYBuf);
    };

    const int L = int(p.seqlen);
    const int64_t dim = p.dim;
    const int b = blockIdx.x / dblocks;
    const int64_t d0 = int64_t(blockIdx.x % dblocks) * CH;
    const int tid = threadIdx.x;
    const int pr = tid / G, g = tid % G;  // chain pair, state group
    const int64_t da = d0 + 2 * pr, db = da + 1;
    const int nchunks = (L + T - 1) / T;
    const int row0 = int(int64_t(b) * dim + d0);
    const bool has_z = p.z != nullptr;
    const io_t* Bg = static_cast<const io_t*>(p.B) + int64_t(b) * L * N;
    const io_t* Cg = static_cast<const io_t*>(p.C) + int64_t(b) * L * N;
    io_t* yy = static_cast<io_t*>(p.y);
    auto chunk_len = [&](int k) { return L - k * T < T ? L - k * T : T; };

    auto issue = [&](int k) {  // one thread
        const uint32_t bc_bytes = uint32_t(chunk_len(k)) * N * C::ES;
        const uint32_t tile_bytes = uint32_t(CH) * T * C::ES;
        uint64_t* br = &bar[k & (S - 1)];
        unsigned char* st = stage(k);
        mbar_arrive_expect_tx(br, (has_z ? 3 : 2) * tile_bytes + 2 * bc_bytes);
        tma_load_2d(st, &tm_u, k * T, row0, br);
        tma_load_2d(st + C::kTile, &tm_d, k * T, row0, br);
        if (has_z) tma_load_2d(st + 2 * C::kTile, &tm_z, k * T, row0, br);
        bulk_g2s(st + 3 * C::kTile, Bg + int64_t(k) * T * N, bc_bytes, br);
        bulk_g2s(st + 3 * C::kTile + C::kRaw, Cg + int64_t(k) * T * N, bc_bytes, br);
    };
    bool copy_failed = false;
    auto wait_chunk = [&](int k) { wait_copy(&bar[k & (S - 1)], uint32_t(k / S) & 1u, copy_failed); };

    // ---- per-element prologue of chunk k, quad item i: (dt, dt*u) ----
    auto elem_prologue = [&](int k, int i) {
        const int sidx = tid + i * NTH;
        if (sidx >= C::NSEG) return;
        const int seg = sidx % C::SEGROW, cc = sidx / C::SEGROW;
        const int64_t dd = d0 + cc;
        const bool live = dd < dim && seg * PV < chunk_len(k);
        const quad_t vd = reinterpret_cast<const quad_t*>(tile(k, 1))[cc * C::SEGROW + seg];
        const quad_t vu = reinterpret_cast<const quad_t*>(tile(k, 0))[cc * C::SEGROW + seg];
        const f32x2 bias2 = splat2((dd < dim && p.delta_bias) ? __ldg(p.delta_bias + dd) : 0.f);
        float* sdf = sdbuf(k);
#pragma unroll
        for (int q = 0; q < PV / 2; ++q) {
            f32x2 dt = add2(get_pair<io_t>(vd, q), bias2);
            if (p.softplus) dt = softplus_pair<io_t>(dt);
            const f32x2 du = mul2(dt, get_pair<io_t>(vu, q));
            float dt0, dt1, du0, du1;
            unpack2(dt, dt0, dt1);
            unpack2(du, du0, du1);
            if (!live) dt0 = dt1 = du0 = du1 = 0.f;
            const int t = seg * PV + 2 * q;
            float* w0 = sdf + (t * NPAIR + pair_col<NPAIR>(t, cc >> 1)) * 4 + (cc & 1);
            float* w1 = sdf + ((t + 1) * NPAIR + pair_col<NPAIR>(t + 1, cc >> 1)) * 4 + (cc & 1);
            w0[0] = dt0;
            w0[2] = du0;
            w1[0] = dt1;
            w1[2] = du1;
        }
    };
    // ---- per-element epilogue of chunk k, quad item i: y ----
    auto elem_epilogue = [&](int k, int i) {
        const int sidx = tid + i * NTH;
        if (sidx >= C::NSEG) return;
        const int seg = sidx % C::SEGROW, cc = sidx / C::SEGROW;
        const int64_t dd = d0 + cc;
        if (dd >= dim || seg * PV >= chunk_len(k)) return;
        f32x2 v[2];
        partial_sums<G, T, C::CH * G>(ybuf(k), cc, seg, v[0], v[1]);
        const quad_t vu = reinterpret_cast<const quad_t*>(tile(k, 0))[cc * C::SEGROW + seg];
        const f32x2 D2 = splat2(p.D ? __ldg(p.D + dd) : 0.f);
        v[0] = fma2(D2, get_pair<io_t>(vu, 0), v[0]);
        v[1] = fma2(D2, get_pair<io_t>(vu, 1), v[1]);
        if (has_z) {
            const quad_t vz = reinterpret_cast<const quad_t*>(tile(k, 2))[cc * C::SEGROW + seg];
            v[0] = gate_pair(v[0], get_pair<io_t>(vz, 0));
            v[1] = gate_pair(v[1], get_pair<io_t>(vz, 1));
        }
        unsigned w[PV * C::ES / 4];
        pack_out<io_t, 2>(v, w);
        *reinterpret_cast<quad_t*>(yy + (int64_t(b) * dim + dd) * L + int64_t(k) * T + seg * PV) =
            *reinterpret_cast<const quad_t*>(w);
    };
    // quad items of this thread handled in 4-step group grp
    auto items_in_group = [&](int i, int grp) { return i * NGRP / SPT == grp; };

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
        fence_proxy_async_smem();
        // chunks kept in flight ahead of the one computed (see the loop)
        for (int k = 0; k < (C::IL ? S - 2 : S - 1) && k < nchunks; ++k) issue(k);
    }

    // A2 pairs across the two chains, per state; states in pairs per chain.
    f32x2 A2p[4], ha[2], hb[2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int n = 4 * g + j;
        const float aa = da < dim ? -expf(__ldg(p.A_log + da * N + n)) * kLog2e : 0.f;
        const float ab = db < dim ? -expf(__ldg(p.A_log + db * N + n)) * kLog2e : 0.f;
        A2p[j] = pack2(aa, ab);
    }
    ha[0] = ha[1] = hb[0] = hb[1] = splat2(0.f);
    __syncthreads();
    if (C::IL && nchunks > 0) {
        wait_chunk(0);
#pragma unroll
        for (int i = 0; i < SPT; ++i) elem_prologue(0, i);
    }
    __syncthreads();

    const int ra = (2 * pr) * G + g, rb = ra + G;  // partial-sum rows of chains a, b

    struct Step {
        ulonglong2 sd;  // (dt_a, dt_b), (du_a, du_b)
        f32x2 aa01, aa23, ab01, ab23;
        f32x2 b01, b23, c01, c23;
    };

    for (int k = 0; k < nchunks; ++k) {
        // Interleaved: refill the stage of chunk k-3 (its epilogue ran before
        // the previous barrier) with chunk k+S-3.  Otherwise the per-element
        // prologue of chunk k runs here, and the stage of chunk k-1 is
        // refilled with chunk k+S-2 after the barrier that follows.
        if (C::IL && tid == 0 && k >= 1 && k + S - 3 < nchunks) {
            fence_proxy_async_smem();
            issue(k + S - 3);
        }
        const bool has_next = C::IL && k + 1 < nchunks, has_prev = C::IL && k >= 1;
        if (has_next) wait_chunk(k + 1);
        if (!C::IL) {
            wait_chunk(k);
#pragma unroll
            for (int i = 0; i < SPT; ++i) elem_prologue(k, i);
            __syncthreads();
            if (tid == 0 && k >= 1 && k + S - 2 < nchunks) {
                fence_proxy_async_smem();
                issue(k + S - 2);
            }
        }
        const int tlen = chunk_len(k);
        const ulonglong2* sd2 = reinterpret_cast<const ulonglong2*>(sdbuf(k));
        const quad_t* rB = reinterpret_cast<const quad_t*>(raw(k, 0));
        const quad_t* rC = reinterpret_cast<const quad_t*>(raw(k, 1));
        float4* y4 = reinterpret_cast<float4*>(ybuf(k));

        auto fetch = [&](int t, Step& st) {
            st.sd = sd2[t * NPAIR + pair_col<NPAIR>(t, pr)];
            float xa[4], xb[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) unpack2(mul2(st.sd.x, A2p[j]), xa[j], xb[j]);
            constexpr bool ACC = sizeof(io_t) == 4;
            st.aa01 = abar_exp2_pair<ACC>(pack2(xa[0], xa[1]));
            st.aa23 = abar_exp2_pair<ACC>(pack2(xa[2], xa[3]));
            st.ab01 = abar_exp2_pair<ACC>(pack2(xb[0], xb[1]));
            st.ab23 = abar_exp2_pair<ACC>(pack2(xb[2], xb[3]));
            const quad_t bq = rB[t * G + g], cq = rC[t * G + g];
            st.b01 = get_pair<io_t>(bq, 0);
            st.b23 = get_pair<io_t>(bq, 1);
            st.c01 = get_pair<io_t>(cq, 0);
            st.c23 = get_pair<io_t>(cq, 1);
        };
        auto update = [&](const Step& st, float& pa, float& pb) {
            float dua, dub;
            unpack2(st.sd.y, dua, dub);
            const f32x2 DA = splat2(dua), DB = splat2(dub);
            ha[0] = fma2(st.aa01, ha[0], mul2(DA, st.b01));
            ha[1] = fma2(st.aa23, ha[1], mul2(DA, st.b23));
            hb[0] = fma2(st.ab01, hb[0], mul2(DB, st.b01));
            hb[1] = fma2(st.ab23, hb[1], mul2(DB, st.b23));
            const f32x2 ya = fma2(st.c23, ha[1], mul2(st.c01, ha[0]));
            const f32x2 yb = fma2(st.c23, hb[1], mul2(st.c01, hb[0]));
            float l, h;
            unpack2(ya, l, h);
            pa = l + h;
            unpack2(yb, l, h);
            pb = l + h;
        };

        if (tlen == T) {
            Step cur;
            fetch(0, cur);
#pragma unroll
            for (int grp = 0; grp < NGRP; ++grp) {
                float pa[4], pb[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int t = 4 * grp + j;
                    Step nxt;
                    if (t + 1 < T) fetch(t + 1, nxt);
                    update(cur, pa[j], pb[j]);
                    if (t + 1 < T) cur = nxt;
                }
                y4[yunit<C::CH * G>(grp, ra)] = make_float4(pa[0], pa[1], pa[2], pa[3]);
                y4[yunit<C::CH * G>(grp, rb)] = make_float4(pb[0], pb[1], pb[2], pb[3]);
                if (C::IL) {
#pragma unroll
                    for (int i = 0; i < SPT; ++i) {
                        if (!items_in_group(i, grp)) continue;
                        if (has_next) elem_prologue(k + 1, i);
                        if (has_prev) elem_epilogue(k - 1, i);
                    }
                }
            }
        } else {
            // ragged last chunk: plain steps, then the neighbours' work
            for (int tt = 0; tt < tlen; tt += 4) {
                float pa[4], pb[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int t = tt + j;
                    pa[j] = pb[j] = 0.f;
                    if (t < tlen) {
                        Step st;
                        fetch(t, st);
                        update(st, pa[j], pb[j]);
                    }
                }
                y4[yunit<C::CH * G>(tt / 4, ra)] = make_float4(pa[0], pa[1], pa[2], pa[3]);
                y4[yunit<C::CH * G>(tt / 4, rb)] = make_float4(pb[0], pb[1], pb[2], pb[3]);
            }
#pragma unroll
            for (int i = 0; i < SPT; ++i) {
                if (has_next) elem_prologue(k + 1, i);
                if (has_prev) elem_epilogue(k - 1, i);
            }
        }
        __syncthreads();
        if (!C::IL) {
#pragma unroll
            for (int i = 0; i < SPT; ++i) elem_epilogue(k, i);
        }
    }
    if (C::IL && nchunks > 0) {
#pragma unroll
        for (int i = 0; i < SPT; ++i) elem_epilogue(nchunks - 1, i);
    }
    if (p.last_state) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int64_t dd = e == 0 ? da : db;
            if (dd >= dim) continue;
            float* out = p.last_state + (int64_t(b) * dim + dd) * N + 4 * g;
            const f32x2* hh = e == 0 ? ha : hb;
            float v0, v1, v2, v3;
            unpack2(hh[0], v0, v1);
            unpack2(hh[1], v2, v3);
            out[0] = v0;
            out[1] = v1;
            out[2] = v2;
            out[3] = v3;
        }
    }
}

// =========================================================================
// Register-prefetch path (rows not 16-byte aligned)
// =========================================================================
template <typename io_t, int NPL_, int G_, int CH_, int T_>
struct RegCfg {
    using io = io_t;
    static constexpr int NPL = NPL_, G = G_, CH = CH_, T = T_;
    static constexpr int NTH = CH * G;
    static constexpr int NP = NPL * G;
    static constexpr int VEC = Io<io_t>::kVec;  // io elements per 16 bytes
    static constexpr int SEGROW = T / VEC;
    static constexpr int NSEG = CH * SEGROW;
    static constexpr int SPT = (NSEG + NTH - 1) / NTH;
    static constexpr int ES = sizeof(io_t);
    static_assert(NPL % 4 == 0 && T % VEC == 0 && T % 4 == 0, "tile shape");
    static_assert((T / 4 & (T / 4 - 1)) == 0, "T/4 must be a power of two");
    static constexpr size_t kStageBytes = size_t(T) * NP * ES;
    static constexpr size_t kStage = 128;
    static constexpr size_t kBf = kStage + 4 * kStageBytes;
    static constexpr size_t kBfBytes = size_t(T) * NP * 4;
    static constexpr size_t kDuBytes = size_t(T) * CH * 16;
    static constexpr size_t kYBytes = size_t(NTH) * T * 4;
    static constexpr size_t kSmem = kBf + 2 * kBfBytes + kDuBytes + kYBytes;
};

// Element-wise load of VEC consecutive io values (zero past L).
template <typename C>
__device__ __forceinline__ uint4 load_seg(const typename C::io* row, int64_t t, int64_t L,
                                          bool valid) {
    unsigned w[4] = {0u, 0u, 0u, 0u};
    if (!valid) return make_uint4(0u, 0u, 0u, 0u);
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

template <typename io_t, int NPL, int G, int CH, int T>
__global__ void __launch_bounds__(CH* G)
    scan_reg_kernel(const ScanArgs p, const int dblocks, const int tma_ok) {
    using C = RegCfg<io_t, NPL, G, CH, T>;
    constexpr int NTH = C::NTH, NP = C::NP, VEC = C::VEC;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    unsigned char* stage = smem + C::kStage;
    float* sB = reinterpret_cast<float*>(smem + C::kBf);
    float* sC = sB + T * NP;
    float4* sdu = reinterpret_cast<float4*>(smem + C::kBf + 2 * C::kBfBytes);
    float* sy = reinterpret_cast<float*>(smem + C::kBf + 2 * C::kBfBytes + C::kDuBytes);

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
    auto stageB = [&](int64_t k) { return stage + size_t(2 * (k & 1)) * C::kStageBytes; };
    auto stageC = [&](int64_t k) { return stage + size_t(2 * (k & 1) + 1) * C::kStageBytes; };
    auto chunk_by_tma = [&](int64_t k) { return tma_ok && (k + 1) * T <= L; };
    auto issue = [&](int64_t k) {  // one thread
        const int64_t off = k * T * N;
        mbar_arrive_expect_tx(&bar[k & 1], 2 * stage_bytes);
        bulk_g2s(stageB(k), Bg + off, stage_bytes, &bar[k & 1]);
        bulk_g2s(stageC(k), Cg + off, stage_bytes, &bar[k & 1]);
    };

    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncthreads();
    if (tid == 0) {
        if (nchunks > 0 && chunk_by_tma(0)) issue(0);
        if (nchunks > 1 && chunk_by_tma(1)) issue(1);
    }
    f32x2 A2[NPL / 2], h[NPL / 2];
    init_state<NPL, G>(p, d, chain_ok, g, A2, h);
    if (p.h0 && chain_ok) load_state<NPL, G>(p.h0 + (int64_t(b) * dim + d) * N, N, g, h);
    const unsigned char* rs = p.reset ? p.reset + int64_t(b) * L : nullptr;

    // slice s = tid + i*NTH is chain s % CH, 16-byte segment s / CH
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
            vd[i] = load_seg<C>(dl + row, t, L, ok);
            vu[i] = load_seg<C>(uu + row, t, L, ok);
            vz[i] = zz ? load_seg<C>(zz + row, t, L, ok) : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    bool copy_failed = false;
    prefetch(0, cur_d, cur_u, cur_z);

    for (int64_t k = 0; k < nchunks; ++k) {
        const int64_t t0 = k * T;
        const int tlen = L - t0 < T ? int(L - t0) : T;

        // ---- phase A ----
        if (chunk_by_tma(k)) {
            wait_copy(&bar[k & 1], uint32_t(k >> 1) & 1u, copy_failed);
            widen_bc<io_t, NP, T, NTH>(stageB(k), stageC(k), sB, sC, N, tid);
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
            const bool live = dd < dim;
            const f32x2 bias2 = splat2((live && p.delta_bias) ? __ldg(p.delta_bias + dd) : 0.f);
#pragma unroll
            for (int q = 0; q < VEC / 2; ++q) {
                f32x2 dt = add2(get_pair<io_t>(cur_d[i], q), bias2);
                if (p.softplus) dt = softplus_pair<io_t>(dt);
                const f32x2 du = mul2(dt, get_pair<io_t>(cur_u[i], q));
                float dt0, dt1, du0, du1;
                unpack2(dt, dt0, dt1);
                unpack2(du, du0, du1);
                const int t = seg * VEC + 2 * q;
                // exponent lane: +inf on a document boundary (Abar = 0)
                float de0 = dt0, de1 = dt1;
                if (rs && live && t < tlen && rs[t0 + t]) de0 = kResetDt;
                if (rs && live && t + 1 < tlen && rs[t0 + t + 1]) de1 = kResetDt;
                if (!(live && t < tlen)) de0 = dt0 = du0 = 0.f;
                if (!(live && t + 1 < tlen)) de1 = dt1 = du1 = 0.f;
                sdu[t * CH + du_col<CH>(t, cc)] = make_float4(de0, de0, du0, du0);
                sdu[(t + 1) * CH + du_col<CH>(t + 1, cc)] = make_float4(de1, de1, du1, du1);
            }
        }
        prefetch(k + 1, nxt_d, nxt_u, nxt_z);
        __syncthreads();

        // ---- phase B ----
        recurrence<sizeof(io_t) == 4, NPL, G, CH, T>(sdu, sB, sC, sy, h, A2, c, g, tid, tlen);
        __syncthreads();
        if (tid == 0 && k + 2 < nchunks && chunk_by_tma(k + 2)) {
            fence_proxy_async_smem();
            issue(k + 2);
        }

        // ---- phase C ----
#pragma unroll
        for (int i = 0; i < C::SPT; ++i) {
            const int sidx = tid + i * NTH;
            if (sidx >= C::NSEG) break;
            const int cc = sidx % CH, seg = sidx / CH;
            const int64_t dd = d0 + cc;
            if (dd >= dim || seg * VEC >= tlen) continue;
            f32x2 v[VEC / 2];
#pragma unroll
            for (int q4 = 0; q4 < VEC / 4; ++q4)
                partial_sums<G, T, CH * G>(sy, cc, seg * (VEC / 4) + q4, v[2 * q4], v[2 * q4 + 1]);
            const f32x2 D2 = splat2(p.D ? __ldg(p.D + dd) : 0.f);
#pragma unroll
            for (int q = 0; q < VEC / 2; ++q) {
                f32x2 o = fma2(D2, get_pair<io_t>(cur_u[i], q), v[q]);
                if (zz) o = gate_pair(o, get_pair<io_t>(cur_z[i], q));
                v[q] = o;
            }
            unsigned w[4];
            pack_out<io_t, VEC / 2>(v, w);
            io_t* row = yy + (int64_t(b) * dim + dd) * L;
            const int64_t t = t0 + seg * VEC;
            if constexpr (C::ES == 4) {
                unsigned* r = reinterpret_cast<unsigned*>(row);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (t + e < L) r[t + e] = w[e];
            } else {
                unsigned short* r = reinterpret_cast<unsigned short*>(row);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (t + e < L) r[t + e] = static_cast<unsigned short>(w[e >> 1] >> (16 * (e & 1)));
            }
        }
#pragma unroll
        for (int i = 0; i < C::SPT; ++i) {
            cur_d[i] = nxt_d[i];
            cur_u[i] = nxt_u[i];
            cur_z[i] = nxt_z[i];
        }
    }
    if (chain_ok && p.last_state) store_state<NPL, G>(p, int64_t(b) * dim + d, g, h);
}

// =========================================================================
// host side
// =========================================================================
int env_int(const char* name) {
    const char* v = getenv(name);
    return v ? atoi(v) : 0;
}

bool al16(const void* q) { return q == nullptr || (reinterpret_cast<uintptr_t>(q) & 15) == 0; }

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(f);
    });
    return fn;
}

// Tensor map of a [rows][L] io array, box = [T steps] x [CH rows].
bool make_map(CUtensorMap* m, const void* base, bool bf16, int64_t rows, int64_t L, int T, int CH) {
    EncodeTiled enc = encode_fn();
    if (!enc) return false;
    const size_t es = bf16 ? 2 : 4;
    const cuuint64_t dims[2] = {cuuint64_t(L), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(L) * es};
    const cuuint32_t box[2] = {cuuint32_t(T), cuuint32_t(CH)};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
               const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename K, typename... Args>
cudaError_t launch(K kern, size_t smem, int64_t blocks, int threads, cudaStream_t stream,
                   Args... args) {
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (err != cudaSuccess) return err;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    kern<<<unsigned(blocks), threads, smem, stream>>>(args...);
    return cudaGetLastError();
}

template <typename io_t, int NPL, int G, int CH>
bool try_tma(const ScanArgs& a, cudaStream_t stream, cudaError_t* err) {
    using C = TmaCfg<io_t, NPL, G, CH>;
    const int64_t es = sizeof(io_t);
    const bool ok = al16(a.u) && al16(a.delta) && al16(a.z) && al16(a.B) && al16(a.C) &&
                    (reinterpret_cast<uintptr_t>(a.y) % (C::PV * es)) == 0 &&
                    (a.seqlen * es) % 16 == 0 && a.batch * a.dim <= 0x7fffffff &&
                    a.seqlen <= 0x7fffffff;
    if (!ok) return false;
    CUtensorMap mu, md, mz;
    const bool bf = sizeof(io_t) == 2;
    const int64_t rows = a.batch * a.dim;
    if (!make_map(&mu, a.u, bf, rows, a.seqlen, C::T, CH) ||
        !make_map(&md, a.delta, bf, rows, a.seqlen, C::T, CH))
        return false;
    if (!make_map(&mz, a.z ? a.z : a.u, bf, rows, a.seqlen, C::T, CH)) return false;
    const int64_t dblocks = (a.dim + CH - 1) / CH;
    *err = launch(scan_tma_kernel<io_t, NPL, G, CH>, C::kSmem, dblocks * a.batch, C::NTH, stream,
                  a, mu, md, mz, int(dblocks));
    return true;
}

template <typename io_t, int NPL, int G, int CH, int T>
cudaError_t launch_reg(const ScanArgs& a, cudaStream_t stream) {
    using C = RegCfg<io_t, NPL, G, CH, T>;
    const int64_t es = sizeof(io_t);
    const int tma_ok = al16(a.B) && al16(a.C) && (a.seqlen * a.dstate * es) % 16 == 0 &&
                       (int64_t(T) * a.dstate * es) % 16 == 0;
    const int64_t dblocks = (a.dim + CH - 1) / CH;
    return launch(scan_reg_kernel<io_t, NPL, G, CH, T>, C::kSmem, dblocks * a.batch, C::NTH,
                  stream, a, int(dblocks), tma_ok);
}

template <typename io_t, int G>
bool try_pair(const ScanArgs& a, cudaStream_t stream, cudaError_t* err) {
    using C = PairCfg<io_t, G>;
    const int64_t es = sizeof(io_t);
    const bool ok = a.dstate == C::N && al16(a.u) && al16(a.delta) && al16(a.z) && al16(a.B) &&
                    al16(a.C) && (reinterpret_cast<uintptr_t>(a.y) % (C::PV * es)) == 0 &&
                    (a.seqlen * es) % 16 == 0 && a.batch * a.dim <= 0x7fffffff &&
                    a.seqlen <= 0x7fffffff;
    if (!ok) return false;
    CUtensorMap mu, md, mz;
    const bool bf = sizeof(io_t) == 2;
    const int64_t rows = a.batch * a.dim;
    if (!make_map(&mu, a.u, bf, rows, a.seqlen, C::T, C::CH) ||
        !make_map(&md, a.delta, bf, rows, a.seqlen, C::T, C::CH) ||
        !make_map(&mz, a.z ? a.z : a.u, bf, rows, a.seqlen, C::T, C::CH))
        return false;
    const int64_t dblocks = (a.dim + C::CH - 1) / C::CH;
    *err = launch(scan_pair_kernel<io_t, G>, C::kSmem, dblocks * a.batch, C::NTH, stream, a, mu,
                  md, mz, int(dblocks));
    return true;
}

// Kernel and tile choice.  Rows that are 16-byte aligned use tensor-map
// kernels: dstate == 16 the single-chain tile with 8 states x 2 threads per
// chain (fastest there; 4 x 4 when there are fewer chains than about 64 per
// SM), dstate in {4, 8, 32, 64, 128} the paired-chain tile,
// other dstate the single-chain tile sized for it.  Unaligned rows use the
// register-prefetch kernel.  MAMBA_SCAN_TILE overrides the choice (1: single
// chain 8x2, 2: single chain 4 states x 4 threads, 3: paired chains) and
// MAMBA_SCAN_PATH=reg forces the register-prefetch kernel; every choice
// computes the same recurrence, and the tests check them against each other.
template <typename io_t, int P, int NPL, int G, int NR, int NE>
bool ws_ok(const ScanArgs& a) {
    using C = WsCfg<io_t, P, NPL, G, NR, NE>;
    const int64_t es = sizeof(io_t);
    return a.dstate == C::NP && al16(a.u) && al16(a.delta) && al16(a.z) && al16(a.B) &&
           al16(a.C) && (reinterpret_cast<uintptr_t>(a.y) % (C::PV * es)) == 0 &&
           (reinterpret_cast<uintptr_t>(a.reset) % 4) == 0 &&
           (a.seqlen * es) % 16 == 0 && a.batch * a.dim <= 0x7fffffff &&
           a.seqlen <= 0x7fffffff;
}

template <typename io_t, int P, int NPL, int G, int NR, int NE, int MINB, int MODE,
          bool FAST = false>
cudaError_t launch_ws(const ScanArgs& a, const SegArgs& sg, cudaStream_t stream) {
    using C = WsCfg<io_t, P, NPL, G, NR, NE>;
    CUtensorMap mu, md, mz;
    const bool bf = sizeof(io_t) == 2;
    const int64_t rows = a.batch * a.dim;
    if (!make_map(&mu, a.u, bf, rows, a.seqlen, C::T, C::CW) ||
        !make_map(&md, a.delta, bf, rows, a.seqlen, C::T, C::CW) ||
        !make_map(&mz, a.z ? a.z : a.u, bf, rows, a.seqlen, C::T, C::CW))
        return cudaErrorInvalidValue;
    const int64_t dblocks = (a.dim + C::CH - 1) / C::CH;
    return launch(scan_ws_kernel<io_t, P, NPL, G, NR, NE, MINB, MODE, FAST>, C::kSmem,
                  dblocks * a.batch * sg.grid_nseg, C::NTH, stream, a, mu, md, mz, int(dblocks),
                  sg);
}

template <typename io_t, int P, int NPL, int G, int NR, int NE, int MINB, bool FAST = false>
bool try_ws(const ScanArgs& a, cudaStream_t stream, cudaError_t* err) {
    if (!ws_ok<io_t, P, NPL, G, NR, NE>(a) || a.seqlen == 0) return false;
    const SegArgs whole{int(a.seqlen), 1, 1, nullptr, nullptr};
    *err = launch_ws<io_t, P, NPL, G, NR, NE, MINB, kScanFull, FAST>(a, whole, stream);
    return *err != cudaErrorInvalidValue;  // tensor map refused: another path
}

// Carry pass of a segmented scan.  For chain c and state n the state entering
// segment 0 is h0 (or zero); the state entering segment s + 1 is
// exp(A_n * sum of dt over s) times the state entering s, plus the end state
// of s from a zero start, which the summary pass left in slot s + 1 (the
// product of the per-step decays exp(dt_t A_n) over a segment is
// exp(A_n * sum dt_t); a document boundary inside s makes the sum +inf and
// the decay 0).  Leaves the state entering segment s in slot s, for every s.
__global__ void __launch_bounds__(256) scan_carry_kernel(const float* A_log, const float* h0,
                                                         SegArgs sg, int64_t chains, int64_t dim,
                                                         int N) {
    const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= chains * N) return;
    const int64_t chain = idx / N, d = chain % dim;
    const int n = int(idx % N);
    const float A2 = fminf(-expf(__ldg(A_log + d * N + n)) * kLog2e, -kA2Max);
    float* slots = sg.hcarry + chain * sg.nseg * N + n;
    float h = h0 ? h0[chain * N + n] : 0.f;
    slots[0] = h;
    for (int s = 0; s + 1 < sg.nseg; ++s) {
        // sdt = +inf when segment s holds a document boundary: decay 0
        h = fmaf(abar_exp2<true>(A2 * sg.sdt[chain * (sg.nseg - 1) + s]), h, slots[(s + 1) * N]);
        slots[(s + 1) * N] = h;
    }
}

// Segments for a scan of few chains.  Splitting costs a summary pass over all
// but the last segment, so it pays only when the unsplit grid leaves at least
// half of the SMs idle; then about 8 CTAs of the dstate-16 tile per SM (two
// waves), each segment at least 512 steps (32 chunks).  Measured on B300 at
// dstate 16: 48 CTAs x L=131072 5.48 -> 1.83 ms (24 segments), 32 CTAs x
// L=32768 1.39 -> 0.42 ms, while 128 CTAs run faster unsplit.
// MAMBA_SCAN_SEGMENTS=n forces n segments (tests).  Returns 1 for no split.
int plan_segments(const ScanArgs& a, int chains_per_cta, int* seg_len) {
    const int64_t L = a.seqlen;
    const int64_t ctas = a.batch * ((a.dim + chains_per_cta - 1) / chains_per_cta);
    int64_t nseg = env_int("MAMBA_SCAN_SEGMENTS");
    if (nseg <= 0) {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            sms <= 0)
            return 1;
        if (2 * ctas > sms) return 1;
        nseg = (8 * int64_t(sms)) / ctas;
        const int64_t by_len = L / 512;
        if (nseg > by_len) nseg = by_len;
    }
    const int64_t max_seg = (L + 15) / 16;
    if (nseg > max_seg) nseg = max_seg;
    if (nseg < 2) return 1;
    const int64_t len = ((L + nseg - 1) / nseg + 15) / 16 * 16;
    *seg_len = int(len);
    return int((L + len - 1) / len);
}

template <typename io_t>
bool try_ws_split(const ScanArgs& a, cudaStream_t stream, const ScanScratch& sc,
                  cudaError_t* err) {
    using C = WsCfg<io_t, 1, 8, 2, 64, 64>;
    if (!ws_ok<io_t, 1, 8, 2, 64, 64>(a) || a.seqlen == 0) return false;
    int seg_len = 0;
    int nseg = plan_segments(a, C::CH, &seg_len);
    if (nseg < 2) return false;
    const int64_t chains = a.batch * a.dim;
    auto rnd = [](size_t x) { return (x + 255) / 256 * 256; };
    auto bytes_for = [&](int ns) {
        return rnd(size_t(chains) * ns * a.dstate * sizeof(float)) +
               rnd(size_t(chains) * (ns - 1) * sizeof(float));
    };
    void* buf = sc.ptr;
    bool owned = false;
    if (buf) {
        // A caller buffer too small for the planner's split takes fewer
        // segments (the planner's choice fits 4 MiB up to ~240 SMs); only a
        // forced segment count that does not fit is an error.
        if (bytes_for(nseg) > sc.bytes && env_int("MAMBA_SCAN_SEGMENTS") <= 0) {
            while (nseg >= 2 && bytes_for(nseg) > sc.bytes) --nseg;
            if (nseg < 2) return false;
            seg_len = int(((a.seqlen + nseg - 1) / nseg + 15) / 16 * 16);
            nseg = int((a.seqlen + seg_len - 1) / seg_len);
        }
        if (bytes_for(nseg) > sc.bytes) {
            *err = cudaErrorMemoryAllocation;
            return true;
        }
    } else {
        // A failed allocation runs the scan unsplit.  It clears the error it
        // set, but only when no error was pending before it.
        const bool pending = cudaPeekAtLastError() != cudaSuccess;
        if (!sc.may_alloc) return false;
        if (scratch_alloc(&buf, bytes_for(nseg), stream) != cudaSuccess) {
            if (!pending) cudaGetLastError();
            return false;
        }
        owned = true;
    }
    const size_t hbytes = rnd(size_t(chains) * nseg * a.dstate * sizeof(float));
    SegArgs sg{seg_len, nseg, nseg - 1, static_cast<float*>(buf),
               reinterpret_cast<float*>(static_cast<char*>(buf) + hbytes)};
    const bool fast = a.z && a.softplus && !a.reset;
    *err = fast ? launch_ws<io_t, 1, 8, 2, 64, 64, 4, kScanSummary, true>(a, sg, stream)
                : launch_ws<io_t, 1, 8, 2, 64, 64, 4, kScanSummary>(a, sg, stream);
    if (*err == cudaSuccess) {
        const int64_t threads = chains * a.dstate;
        scan_carry_kernel<<<unsigned((threads + 255) / 256), 256, 0, stream>>>(
            a.A_log, a.h0, sg, chains, a.dim, a.dstate);
        *err = cudaGetLastError();
    }
    if (*err == cudaSuccess) {
        sg.grid_nseg = nseg;
        *err = fast ? launch_ws<io_t, 1, 8, 2, 64, 64, 4, kScanFull, true>(a, sg, stream)
                    : launch_ws<io_t, 1, 8, 2, 64, 64, 4, kScanFull>(a, sg, stream);
    }
    if (owned) {
        const cudaError_t ferr = scratch_free(buf, stream);
        if (*err == cudaSuccess) *err = ferr;
    }
    return true;
}

bool force_reg() {
    const char* v = getenv("MAMBA_SCAN_PATH");
    return v && v[0] == 'r';
}

template <typename io_t>
bool try_pair_n(const ScanArgs& a, cudaStream_t stream, cudaError_t* err) {
    switch (a.dstate) {
        case 4: return try_pair<io_t, 1>(a, stream, err);
        case 8: return try_pair<io_t, 2>(a, stream, err);
        case 16: return try_pair<io_t, 4>(a, stream, err);
        case 32: return try_pair<io_t, 8>(a, stream, err);
        case 64: return try_pair<io_t, 16>(a, stream, err);
        case 128: return try_pair<io_t, 32>(a, stream, err);
        default: return false;
    }
}

template <typename io_t, int NPL, int G, int CH, int TREG>
cudaError_t run(const ScanArgs& a, cudaStream_t stream, bool pair_first) {
    cudaError_t err = cudaSuccess;
    // The paired and tensor-map tiles take no initial state or reset mask:
    // those calls go to the register-prefetch kernel.
    if (!force_reg() && !a.h0 && !a.reset) {
        if (pair_first && try_pair_n<io_t>(a, stream, &err)) return err;
        if (try_tma<io_t, NPL, G, CH>(a, stream, &err)) return err;
    }
    return launch_reg<io_t, NPL, G, CH, TREG>(a, stream);
}

template <typename io_t>
cudaError_t dispatch(const ScanArgs& a, cudaStream_t stream, const ScanScratch& sc) {
    const int N = a.dstate;
    const int tile = env_int("MAMBA_SCAN_TILE");
    const bool pair = tile == 3 || (tile == 0 && N != 16);
    if (N <= 4) return run<io_t, 4, 1, 64, 8>(a, stream, pair);
    if (N <= 8) return run<io_t, 4, 2, 32, 16>(a, stream, pair);
    if (N <= 16) {
        // Few chains (long sequences, small batch): more threads per chain.
        const bool few = a.batch * a.dim < 148 * 64;
        cudaError_t err = cudaSuccess;
        // Few chains and a long sequence: split the sequence (see try_ws_split).
        if ((tile == 0 || tile == 4) && N == 16 && !force_reg() &&
            try_ws_split<io_t>(a, stream, sc, &err))
            return err;
        const bool fast = a.z && a.softplus && !a.reset;
        if ((tile == 4 || tile == 0) && N == 16 && !force_reg() && fast &&
            try_ws<io_t, 1, 8, 2, 64, 64, 4, true>(a, stream, &err))
            return err;
        if ((tile == 4 || tile == 0) && N == 16 && !force_reg() &&
            try_ws<io_t, 1, 8, 2, 64, 64, 4>(a, stream, &err))
            return err;
        if (tile == 5 && N == 16 && !force_reg() && try_ws<io_t, 2, 8, 2, 64, 64, 2>(a, stream, &err))
            return err;
        if (tile == 6 && N == 16 && !force_reg() && try_ws<io_t, 2, 4, 4, 64, 64, 4>(a, stream, &err))
            return err;
        if (tile == 7 && N == 16 && !force_reg() && try_ws<io_t, 1, 4, 4, 128, 64, 4>(a, stream, &err))
            return err;
        if (tile == 8 && N == 16 && !force_reg() && fast &&
            try_ws<io_t, 1, 8, 2, 32, 32, 8, true>(a, stream, &err))
            return err;
        if (tile == 8 && N == 16 && !force_reg() && try_ws<io_t, 1, 8, 2, 32, 32, 8>(a, stream, &err))
            return err;
        // dstate 16 falls back to the 8-state x 2-lane arrangement of the tile
        // above, so that both sum C.h in the same order.
        if (tile == 2 || (tile == 0 && few && N != 16)) return run<io_t, 4, 4, 16, 32>(a, stream, false);
        return run<io_t, 8, 2, 32, 16>(a, stream, pair);
    }
    if (N <= 32) return run<io_t, 4, 8, 8, 32>(a, stream, pair);
    if (N == 64 && tile == 4 && !force_reg()) {
        // 16 states x 4 lanes per chain, 16 chains per CTA, two CTAs per SM.
        // Measured at 2 x 2048 x 8192 fp32: 1.85 ms against 0.97 ms for the
        // paired tile -- under one recurrence warp per scheduler cannot hide
        // a 16-state step's latency -- so it is a selectable variant only.
        cudaError_t err = cudaSuccess;
        if (try_ws<io_t, 1, 16, 4, 64, 64, 2>(a, stream, &err)) return err;
    }
    if (N <= 64) return run<io_t, 4, 16, 4, 16>(a, stream, pair);
    if (N <= 128) return run<io_t, 4, 32, 2, 16>(a, stream, pair);
    return run<io_t, 8, 32, 2, 8>(a, stream, pair);
}

}  // namespace

cudaError_t launch_scan_fwd(const ScanArgs& a, bool bf16, cudaStream_t stream,
                            const ScanScratch& sc) {
    return bf16 ? dispatch<__nv_bfloat16>(a, stream, sc) : dispatch<float>(a, stream, sc);
}

// Test hook: one thread waits, with `limit` polls, on an mbarrier that nothing
// ever arrives on, and records the give-up in the error word exactly as the
// scans' bounded copy waits do.  Nothing is copied, so nothing is in flight
// when the kernel ends.
__global__ void bounded_wait_probe_kernel(uint32_t limit) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait_n(&bar, 0u, limit)) atomicOr(&g_scan_error, kErrWaitTimeout);
}

cudaError_t launch_bounded_wait_probe(uint32_t limit, cudaStream_t stream) {
    bounded_wait_probe_kernel<<<1, 32, 0, stream>>>(limit);
    return cudaGetLastError();
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
