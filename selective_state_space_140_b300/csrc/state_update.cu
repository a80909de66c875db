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
#include <cstdlib>

#include "common.cuh"
#include "launch_dep.cuh"

namespace mamba {

// Device error word of the decode kernels' bounded waits; mamba_device_status
// reads and clears it together with the scan's.
__device__ unsigned int g_decode_error;

namespace {

// The grid covers each batch row with `bpr` blocks of 256 / G channels, so a
// thread finds its (b, d) from its block with one division per block (the
// per-thread 64-bit division by dim cost more than the whole state update).
template <typename io_t, int NPL, int G, bool VEC>
__global__ void __launch_bounds__(256) state_update_kernel(StateUpdateArgs p, uint32_t bpr) {
    const uint32_t bi = blockIdx.x / bpr;  // the same for the whole block
    const int64_t b = bi;
    const int64_t d = int64_t(blockIdx.x - bi * bpr) * (256 / G) + threadIdx.x / G;
    const int g = int(threadIdx.x % G);
    // Whole G-lane groups are inside or outside together (G divides 32 and the
    // block size), so the shuffles below never mix live and dead lanes.
    if (d >= p.dim) return;
    const int64_t chain = b * p.dim + d;
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
    const int64_t bpr = (a.dim + 256 / G - 1) / (256 / G);  // blocks per batch row
    const int64_t blocks = a.batch * bpr;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const bool vec = (a.dstate % 4 == 0) && (a.dstate == NPL * G) &&
                     (reinterpret_cast<uintptr_t>(a.state) % 16 == 0);
    if (vec)
        state_update_kernel<io_t, NPL, G, true><<<unsigned(blocks), 256, 0, stream>>>(a, uint32_t(bpr));
    else
        state_update_kernel<io_t, NPL, G, false><<<unsigned(blocks), 256, 0, stream>>>(a, uint32_t(bpr));
    return cudaGetLastError();
}

// ---- bulk-copy ring path ------------------------------------------------
// One 16-byte state access per thread keeps too few bytes in flight for the
// HBM.  Here persistent CTAs of 256 threads walk tiles of TC = 4096 / N
// chains (16 KB of state) of one channel block: CTA c owns channel block
// c mod T1 (and every T1-th block after it when there are more blocks than
// CTAs) and, within it, the batch rows c / T1, c / T1 + R, ...  A_log, the
// bias and D do not depend on the batch row, so A * log2 e, the bias and D of
// the thread's chains stay in registers while the CTA walks its batch rows,
// and the copies carry only what changes per tile: thread 0 keeps S tiles in
// flight as bulk copies (cp.async.bulk: the state rows and the tile's dt, x
// and z) into a shared-memory ring completed on mbarriers.  B and C of the
// batch row are loaded before a tile's copy is waited for; each pass is then
// arithmetic on shared memory, and the new state is stored straight to
// global memory.
constexpr int kRingTileBytes = 16384;

// Stage layout: state rows | dt | x | z (each a 16-byte multiple).
template <typename io_t, int G>
struct RingCfg {
    static constexpr int NPL = 4, N = NPL * G, TC = kRingTileBytes / (N * 4), CPP = 256 / G;
    static constexpr int PASSES = TC / CPP, ES = sizeof(io_t), S = 3;
    static constexpr int kIoBytes = TC * ES;  // dt, x or z of one tile
    static constexpr int kDt = kRingTileBytes, kX = kDt + kIoBytes, kZ = kX + kIoBytes;
    static constexpr int kStage = (kZ + kIoBytes + 127) / 128 * 128;
    static constexpr int kSmem = 128 + S * kStage;
    static_assert(PASSES * CPP == TC && kIoBytes % 16 == 0, "tile shape");
};

template <typename io_t, int G>
__global__ void __launch_bounds__(256, 4) state_update_ring_kernel(StateUpdateArgs p, int T1,
                                                                   int R) {
    using C = RingCfg<io_t, G>;
    constexpr int N = C::N, TC = C::TC, CPP = C::CPP, PASSES = C::PASSES, S = C::S;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    auto stage = [&](int st) { return smem + 128 + st * C::kStage; };
    const int tid = threadIdx.x, g = tid % G, cl = tid / G;
    const bool has_z = p.z != nullptr;

    // this CTA's tiles j = 0 .. njobs-1: channel block cb0 + (j / nb) * T1,
    // batch row b0 + (j % nb) * R
    const int64_t tpr = p.dim / TC;  // channel blocks per batch row
    const int64_t cb0 = blockIdx.x % T1, b0 = blockIdx.x / T1;
    const int64_t nb = b0 < p.batch ? (p.batch - b0 + R - 1) / R : 0;
    const int64_t ncb = cb0 < tpr ? (tpr - cb0 + T1 - 1) / T1 : 0;
    const int64_t njobs = nb * ncb;
    auto tile_cb = [&](int64_t j) { return cb0 + (j / nb) * T1; };
    auto tile_b = [&](int64_t j) { return b0 + (j % nb) * R; };
    auto issue = [&](int64_t j, int st) {  // thread 0
        const int64_t c0 = tile_b(j) * p.dim + tile_cb(j) * TC;  // first chain of the tile
        unsigned char* sp = stage(st);
        mbar_arrive_expect_tx(&bar[st], kRingTileBytes + (has_z ? 3 : 2) * C::kIoBytes);
        bulk_g2s(sp, p.state + c0 * N, kRingTileBytes, &bar[st]);
        bulk_g2s(sp + C::kDt, static_cast<const io_t*>(p.dt) + c0, C::kIoBytes, &bar[st]);
        bulk_g2s(sp + C::kX, static_cast<const io_t*>(p.x) + c0, C::kIoBytes, &bar[st]);
        if (has_z) bulk_g2s(sp + C::kZ, static_cast<const io_t*>(p.z) + c0, C::kIoBytes, &bar[st]);
    };
    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);  // (S <= 16 fit in 128 bytes)
        fence_mbar_init();
    }
    // Launched as a programmatic dependent of the previous kernel on the
    // stream (a decode loop's previous step), this CTA may start while that
    // kernel drains: nothing above reads or writes global memory, and the wait
    // returns once the previous grid has completed and its writes are
    // visible.  The next launch may then be scheduled as this grid's CTAs
    // exit.  Without the launch attribute both are no-ops.
    grid_dependency_wait();
    grid_launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < S && s < njobs; ++s) issue(s, s);
    }
    __syncthreads();

    const unsigned lane = tid & 31u;
    const unsigned gmask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (lane / G * G));
    bool failed = false;
    // per-channel parameters of the thread's chain in each pass, for the
    // current channel block (A2 = A * log2 e, A = -exp(A_log) = -2^(A_log log2 e))
    float A2[PASSES][4], bias[PASSES], Dd[PASSES];
    float bias_e = 0.f, D_e = 0.f;  // of the chain whose per-chain work this lane does (G >= PASSES)
    int64_t cur_cb = -1;
    for (int64_t j = 0; j < njobs; ++j) {
        const int st = int(j % S);
        const int64_t b = tile_b(j), cb = tile_cb(j);
        if (cb != cur_cb) {
            cur_cb = cb;
#pragma unroll
            for (int ps = 0; ps < PASSES; ++ps) {
                const int64_t d = cb * TC + ps * CPP + cl;
                const float4 al = __ldg(reinterpret_cast<const float4*>(p.A_log + d * N) + g);
                const float av[4] = {al.x, al.y, al.z, al.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) A2[ps][i] = -ex2_approx(av[i] * kLog2e) * kLog2e;
                bias[ps] = p.dt_bias ? __ldg(p.dt_bias + d) : 0.f;
                Dd[ps] = p.D ? __ldg(p.D + d) : 0.f;
            }
            if constexpr (G >= PASSES) {
                const int64_t d = cb * TC + (g < PASSES ? g : 0) * CPP + cl;
                bias_e = p.dt_bias ? __ldg(p.dt_bias + d) : 0.f;
                D_e = p.D ? __ldg(p.D + d) : 0.f;
            }
        }
        // ---- B and C of the batch row first: they do not depend on the copy ----
        float Bv[4], Cv[4];
        {
            const io_t* Bb = static_cast<const io_t*>(p.B) + b * N + g * 4;
            const io_t* Cb = static_cast<const io_t*>(p.C) + b * N + g * 4;
            if constexpr (sizeof(io_t) == 2) {
                const uint2 wb = __ldg(reinterpret_cast<const uint2*>(Bb));
                const uint2 wc = __ldg(reinterpret_cast<const uint2*>(Cb));
                Bv[0] = __uint_as_float(wb.x << 16); Bv[1] = __uint_as_float(wb.x & 0xffff0000u);
                Bv[2] = __uint_as_float(wb.y << 16); Bv[3] = __uint_as_float(wb.y & 0xffff0000u);
                Cv[0] = __uint_as_float(wc.x << 16); Cv[1] = __uint_as_float(wc.x & 0xffff0000u);
                Cv[2] = __uint_as_float(wc.y << 16); Cv[3] = __uint_as_float(wc.y & 0xffff0000u);
            } else {
                const float4 vb = __ldg(reinterpret_cast<const float4*>(Bb));
                const float4 vc = __ldg(reinterpret_cast<const float4*>(Cb));
                Bv[0] = vb.x; Bv[1] = vb.y; Bv[2] = vb.z; Bv[3] = vb.w;
                Cv[0] = vc.x; Cv[1] = vc.y; Cv[2] = vc.z; Cv[3] = vc.w;
            }
        }
        if (!mbar_wait_n(&bar[st], uint32_t(j / S) & 1u,
                         failed ? kWaitLimitAfterFailure : kWaitLimit)) {
            failed = true;
            atomicOr(&g_decode_error, kErrWaitTimeout);
        }
        const unsigned char* sp = stage(st);
        const io_t* sdt = reinterpret_cast<const io_t*>(sp + C::kDt);
        const io_t* sx = reinterpret_cast<const io_t*>(sp + C::kX);
        const io_t* sz = reinterpret_cast<const io_t*>(sp + C::kZ);
        const int64_t c0 = b * p.dim + cb * TC;
        if constexpr (G >= PASSES) {
            // Lane g < PASSES of a chain group does the per-chain work of pass g
            // (dt, dt * x, skip, gate, store); dt and dt * x reach the group's
            // lanes by shuffles, and every lane updates its 4 states of each pass.
            const int ge = g < PASSES ? g : 0, local_e = ge * CPP + cl;
            const float raw = float(sdt[local_e]) + bias_e;
            const float x_e = float(sx[local_e]);
            const float dt_e = !p.softplus ? raw : sizeof(io_t) == 2 ? softplus_fast(raw)
                                                                       : softplus_accurate(raw);
            const float dx_e = dt_e * x_e;
            float acc[PASSES];
#pragma unroll
            for (int ps = 0; ps < PASSES; ++ps) {
                const int local = ps * CPP + cl;
                const float dt = __shfl_sync(gmask, dt_e, ps, G);
                const float dx = __shfl_sync(gmask, dx_e, ps, G);
                const float4 hv = reinterpret_cast<const float4*>(sp)[local * G + g];
                float h[4] = {hv.x, hv.y, hv.z, hv.w};
                float a = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    h[i] = fmaf(ex2_approx(dt * A2[ps][i]), h[i], dx * Bv[i]);
                    a = fmaf(Cv[i], h[i], a);
                }
                reinterpret_cast<float4*>(p.state + (c0 + local) * N)[g] =
                    make_float4(h[0], h[1], h[2], h[3]);
                acc[ps] = a;
            }
#pragma unroll
            for (int ps = 0; ps < PASSES; ++ps)
#pragma unroll
                for (int off = G / 2; off > 0; off /= 2)
                    acc[ps] += __shfl_xor_sync(gmask, acc[ps], off, G);
            if (g < PASSES) {
                float tot = acc[0];
#pragma unroll
                for (int ps = 1; ps < PASSES; ++ps)
                    if (g == ps) tot = acc[ps];
                if (p.D) tot = fmaf(D_e, x_e, tot);
                if (has_z) tot *= silu_fast(float(sz[local_e]));
                Io<io_t>::store(static_cast<io_t*>(p.out) + c0 + local_e, tot);
            }
        } else {
#pragma unroll
        for (int ps = 0; ps < PASSES; ++ps) {
            const int local = ps * CPP + cl;
            const int64_t chain = c0 + local;
            const float4 hv = reinterpret_cast<const float4*>(sp)[local * G + g];
            const float raw = float(sdt[local]) + bias[ps];
            const float x = float(sx[local]);
            const float dt = !p.softplus ? raw : sizeof(io_t) == 2 ? softplus_fast(raw)
                                                                     : softplus_accurate(raw);
            const float dx = dt * x;
            float h[4] = {hv.x, hv.y, hv.z, hv.w};
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                h[i] = fmaf(ex2_approx(dt * A2[ps][i]), h[i], dx * Bv[i]);
                acc = fmaf(Cv[i], h[i], acc);
            }
            reinterpret_cast<float4*>(p.state + chain * N)[g] = make_float4(h[0], h[1], h[2], h[3]);
#pragma unroll
            for (int off = G / 2; off > 0; off /= 2) acc += __shfl_xor_sync(gmask, acc, off, G);
            if (g == 0) {
                if (p.D) acc = fmaf(Dd[ps], x, acc);
                if (has_z) acc *= silu_fast(float(sz[local]));
                Io<io_t>::store(static_cast<io_t*>(p.out) + chain, acc);
            }
        }
        }
        __syncthreads();  // every thread is done with this stage
        if (tid == 0 && j + S < njobs) {
            fence_proxy_async_smem();
            issue(j + S, st);
        }
    }
}

// The ring needs whole tiles inside batch rows (dim a multiple of TC) and
// 16-byte aligned state, A_log, dt, x, z and B/C rows of 4 elements.
template <typename io_t, int G>
bool try_ring(const StateUpdateArgs& a, cudaStream_t stream, cudaError_t* err) {
    using C = RingCfg<io_t, G>;
    auto al = [](const void* q, size_t n) {
        return q == nullptr || reinterpret_cast<uintptr_t>(q) % n == 0;
    };
    if (a.dstate != C::N || a.dim % C::TC != 0 || !al(a.state, 16) || !al(a.A_log, 16) ||
        !al(a.dt, 16) || !al(a.x, 16) || !al(a.z, 16) || !al(a.B, 4 * C::ES) ||
        !al(a.C, 4 * C::ES) || a.batch > 0x7fffffff)
        return false;
    auto kern = state_update_ring_kernel<io_t, G>;
    // SM count, shared-memory attribute and resident CTAs: once per device
    static LaunchShapeCache shape;
    int sms = 0, per_sm = 0;
    if (!cached_launch_shape(
            shape,
            [&](int* s, int* r) {
                int dev = 0;
                return cudaGetDevice(&dev) == cudaSuccess &&
                       cudaDeviceGetAttribute(s, cudaDevAttrMultiProcessorCount, dev) ==
                           cudaSuccess &&
                       cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            C::kSmem) == cudaSuccess &&
                       cudaOccupancyMaxActiveBlocksPerMultiprocessor(r, kern, 256, C::kSmem) ==
                           cudaSuccess;
            },
            &sms, &per_sm))
        return false;
    // One persistent CTA per slot: T1 channel-block columns x R batch strides.
    const int64_t slots = int64_t(sms) * per_sm, tpr = a.dim / C::TC;
    int64_t T1 = tpr, R = 1;
    if (tpr <= slots) {
        R = slots / tpr;
        if (R > a.batch) R = a.batch;
    } else {
        T1 = slots;
    }
    // Programmatic dependent launch (MAMBA_DECODE_PDL=0 turns it off): the
    // CTAs of consecutive decode steps overlap the previous step's tail.
    *err = launch_dependent(kern, dim3(unsigned(T1 * R)), dim3(256), C::kSmem, stream,
                            "MAMBA_DECODE_PDL", a, int(T1), int(R));
    return true;
}

template <typename io_t>
cudaError_t dispatch(const StateUpdateArgs& a, cudaStream_t stream) {
    const int N = a.dstate;
    cudaError_t err = cudaSuccess;
    const char* path = getenv("MAMBA_DECODE_PATH");
    if (!(path && path[0] == 'p')) {  // MAMBA_DECODE_PATH=plain: one access per thread
        if (N == 4 && try_ring<io_t, 1>(a, stream, &err)) return err;
        if (N == 8 && try_ring<io_t, 2>(a, stream, &err)) return err;
        if (N == 16 && try_ring<io_t, 4>(a, stream, &err)) return err;
        if (N == 32 && try_ring<io_t, 8>(a, stream, &err)) return err;
        if (N == 64 && try_ring<io_t, 16>(a, stream, &err)) return err;
        if (N == 128 && try_ring<io_t, 32>(a, stream, &err)) return err;
    }
    if (N <= 4) return launch<io_t, 4, 1>(a, stream);
    if (N <= 8) return launch<io_t, 4, 2>(a, stream);
    if (N <= 16) return launch<io_t, 4, 4>(a, stream);
    if (N <= 32) return launch<io_t, 4, 8>(a, stream);
    if (N <= 64) return launch<io_t, 4, 16>(a, stream);
    if (N <= 128) return launch<io_t, 4, 32>(a, stream);
    return launch<io_t, 8, 32>(a, stream);
}

}  // namespace

cudaError_t read_and_clear_decode_error(unsigned int* word) {
    const cudaError_t err = cudaMemcpyFromSymbol(word, g_decode_error, sizeof(unsigned int));
    if (err != cudaSuccess) return err;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_decode_error, &zero, sizeof(unsigned int));
}

cudaError_t launch_state_update(const StateUpdateArgs& a, bool bf16, cudaStream_t stream) {
    return bf16 ? dispatch<__nv_bfloat16>(a, stream) : dispatch<float>(a, stream);
}

}  // namespace mamba
