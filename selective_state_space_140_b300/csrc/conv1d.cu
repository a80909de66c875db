// Causal depthwise conv1d + SiLU in front of the scan, sm_103a.
//
// The Mamba block runs its x branch through a short per-channel convolution
// before the scan (luzhipeng.com tutorial, step 2: nn.Conv1d with
// kernel_size = d_conv, padding = d_conv - 1, groups = d_model;
// highthink.cn "Mamba 整体架构": a causal Conv1D followed by SiLU).  For every
// row (b, d) and step t
//   out[t] = SiLU(bias[d] + sum_k w[d][k] * xin(t - (width-1) + k))
// where xin(s) = x[s] for s >= 0 and the caller's conv state (the last
// width-1 inputs of a previous block, oldest first) or zero before the row.
//
// The work is one read of x and one write of out per element (HBM bound).
// Fast path: one thread per 16-byte vector of V outputs; the width-1 inputs
// before the vector come from the previous lane's registers (a shuffle), or
// for the first lane of a warp, from a second load of the previous vector
// (an L1/L2 hit) or the conv state.  Rows of any length and other alignments
// take a scalar path: one thread per output.  The decode step (one token per
// row) shifts the conv state in place.
#include "common.cuh"
#include "launch_dep.cuh"

namespace mamba {
namespace {

template <typename io_t>
struct Vec;
template <>
struct Vec<float> {
    static constexpr int V = 4;
    static __device__ __forceinline__ void unpack(const uint4& r, float* v) {
        v[0] = __uint_as_float(r.x); v[1] = __uint_as_float(r.y);
        v[2] = __uint_as_float(r.z); v[3] = __uint_as_float(r.w);
    }
    static __device__ __forceinline__ uint4 pack(const float* v) {
        return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                          __float_as_uint(v[3]));
    }
};
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int V = 8;
    static __device__ __forceinline__ void unpack(const uint4& r, float* v) {
        const unsigned w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    static __device__ __forceinline__ uint4 pack(const float* v) {
        unsigned w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 p = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<const unsigned*>(&p);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

__device__ __forceinline__ float act(float pre, bool silu) {
    return silu ? pre * rcp_approx(1.f + ex2_approx(-pre * kLog2e)) : pre;
}

struct ConvArgs {
    const void* x;
    const float* w;      // [dim][width]
    const float* bias;   // [dim] or null
    const void* st_in;   // [rows][width-1] or null
    void* out;
    void* st_out;        // [rows][width-1] or null
    int64_t rows, dim, L;
    int width;
    bool silu;
};

__device__ __forceinline__ uint4 ldg16(const void* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

// One thread per V-element vector of a row (L % V == 0, 16-byte aligned rows,
// K - 1 <= V).  Each warp takes segments of 32 * U consecutive vectors of one
// row (one division per segment, the channel's taps loaded once per segment)
// and issues all U loads of a segment before using any.  Within a group of 32
// lane l's previous inputs are lane l-1's vector; lane 0 takes lane 31's
// vector of the previous group, and in the first group it reloads its
// predecessor (an L1/L2 hit) unless the segment starts the row.  Launched as
// a programmatic dependent of the kernel before it on the stream.
template <typename io_t, int K, int U>
__global__ void __launch_bounds__(256) conv_vec_kernel(const ConvArgs a) {
    constexpr int V = Vec<io_t>::V, H = K - 1, HP = H > 0 ? H : 1, SEG = 32 * U;
    grid_dependency_wait();  // before the first global memory access
    grid_launch_dependents();
    const io_t* x = static_cast<const io_t*>(a.x);
    io_t* out = static_cast<io_t*>(a.out);
    const io_t* st_in = static_cast<const io_t*>(a.st_in);
    io_t* st_out = static_cast<io_t*>(a.st_out);
    const int64_t nv_row = a.L / V;
    const int64_t nseg_row = (nv_row + SEG - 1) / SEG, nseg = a.rows * nseg_row;
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x / 32);
    for (int64_t sg = int64_t(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32; sg < nseg;
         sg += nwarps) {
        const int64_t row = sg / nseg_row, v0 = (sg - row * nseg_row) * SEG;
        const int64_t d = row % a.dim;
        const io_t* xr = x + row * a.L;
        io_t* orow = out + row * a.L;
        float w[K];
#pragma unroll
        for (int k = 0; k < K; ++k) w[k] = __ldg(a.w + d * K + k);
        const float bias = a.bias ? __ldg(a.bias + d) : 0.f;
        uint4 raw[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t vr = v0 + u * 32 + lane;
            raw[u] = vr < nv_row ? ldg16(xr + vr * V) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t vr = v0 + u * 32 + lane;
            const int src = lane == 0 ? 31 : lane - 1;
            // lane 0 reads lane 31, which supplies its vector of the previous group
            // (no other lane reads lane 31); the other lanes read lane - 1's vector
            const uint4 cur = raw[u], prv = raw[u > 0 ? u - 1 : 0];
            const bool take_prv = lane == 31 && u > 0;
            uint4 pr;
            pr.x = __shfl_sync(0xffffffffu, take_prv ? prv.x : cur.x, src);
            pr.y = __shfl_sync(0xffffffffu, take_prv ? prv.y : cur.y, src);
            pr.z = __shfl_sync(0xffffffffu, take_prv ? prv.z : cur.z, src);
            pr.w = __shfl_sync(0xffffffffu, take_prv ? prv.w : cur.w, src);
            if (vr >= nv_row) continue;
            if (lane == 0 && u == 0 && vr > 0) pr = ldg16(xr + (vr - 1) * V);
            float win[HP + V];
            Vec<io_t>::unpack(cur, win + HP);
            if constexpr (H > 0) {
                if (vr > 0) {
                    float pv[V];
                    Vec<io_t>::unpack(pr, pv);
#pragma unroll
                    for (int i = 0; i < H; ++i) win[HP - H + i] = pv[V - H + i];
                } else {
#pragma unroll
                    for (int i = 0; i < H; ++i)
                        win[HP - H + i] = st_in ? Io<io_t>::load(st_in + row * H + i) : 0.f;
                }
            }
            float o[V];
#pragma unroll
            for (int j = 0; j < V; ++j) {
                float pre = bias;
#pragma unroll
                for (int k = 0; k < K; ++k) pre = fmaf(w[k], win[HP - H + j + k], pre);
                o[j] = act(pre, a.silu);
            }
            *reinterpret_cast<uint4*>(orow + vr * V) = Vec<io_t>::pack(o);
            if constexpr (H > 0) {
                if (st_out && vr == nv_row - 1) {
#pragma unroll
                    for (int i = 0; i < H; ++i)
                        Io<io_t>::store(st_out + row * H + i, win[HP + V - H + i]);
                }
            }
        }
    }
}

// xin(s) of one row: the input for s >= 0, else the conv state (or zero)
template <typename io_t>
__device__ __forceinline__ float conv_in(const io_t* xr, const io_t* st, int H, int64_t s) {
    if (s >= 0) return Io<io_t>::load(xr + s);
    return st ? Io<io_t>::load(st + H + s) : 0.f;
}

// One thread per output element; any length, alignment and width.
template <typename io_t>
__global__ void __launch_bounds__(256) conv_scalar_kernel(const ConvArgs a) {
    const io_t* x = static_cast<const io_t*>(a.x);
    const io_t* st_in = static_cast<const io_t*>(a.st_in);
    io_t* out = static_cast<io_t*>(a.out);
    io_t* st_out = static_cast<io_t*>(a.st_out);
    const int K = a.width, H = K - 1;
    const int64_t total = a.rows * a.L;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < total; e += stride) {
        const int64_t row = e / a.L, t = e % a.L, d = row % a.dim;
        const io_t* xr = x + row * a.L;
        const io_t* st = st_in ? st_in + row * H : nullptr;
        float pre = a.bias ? __ldg(a.bias + d) : 0.f;
        for (int k = 0; k < K; ++k) pre = fmaf(__ldg(a.w + d * K + k), conv_in(xr, st, H, t - H + k), pre);
        Io<io_t>::store(out + e, act(pre, a.silu));
        if (st_out && t == a.L - 1)
            for (int i = 0; i < H; ++i)
                Io<io_t>::store(st_out + row * H + i, conv_in(xr, st, H, a.L - H + i));
    }
}

// seqlen 0: the final state is the initial state (or zeros)
template <typename io_t>
__global__ void __launch_bounds__(256) conv_state_copy_kernel(const ConvArgs a) {
    const int H = a.width - 1;
    const io_t* st_in = static_cast<const io_t*>(a.st_in);
    io_t* st_out = static_cast<io_t*>(a.st_out);
    const int64_t total = a.rows * H;
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
         e += int64_t(gridDim.x) * blockDim.x)
        Io<io_t>::store(st_out + e, st_in ? Io<io_t>::load(st_in + e) : 0.f);
}

// Decode: one token per row; the conv state [rows][width-1] shifts in place.
template <typename io_t>
__global__ void __launch_bounds__(256) conv_update_kernel(void* state_, const void* x_,
                                                          const float* w, const float* bias,
                                                          void* out_, int64_t rows, int64_t dim,
                                                          int K, bool silu) {
    io_t* state = static_cast<io_t*>(state_);
    const io_t* x = static_cast<const io_t*>(x_);
    io_t* out = static_cast<io_t*>(out_);
    const int H = K - 1;
    for (int64_t row = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; row < rows;
         row += int64_t(gridDim.x) * blockDim.x) {
        const int64_t d = row % dim;
        io_t* st = state + row * H;
        const float xv = Io<io_t>::load(x + row);
        float pre = bias ? __ldg(bias + d) : 0.f;
        for (int k = 0; k < H; ++k) pre = fmaf(__ldg(w + d * K + k), Io<io_t>::load(st + k), pre);
        pre = fmaf(__ldg(w + d * K + H), xv, pre);
        Io<io_t>::store(out + row, act(pre, silu));
        for (int k = 0; k + 1 < H; ++k) st[k] = st[k + 1];
        if (H > 0) st[H - 1] = x[row];
    }
}

int grid_for(int64_t work, int per_block) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (work + per_block - 1) / per_block;
    const int64_t cap = int64_t(sms) * 16;  // grid-stride beyond 16 blocks of 256 per SM
    return int(want < 1 ? 1 : (want < cap ? want : cap));
}

bool al16(const void* q) { return q == nullptr || (reinterpret_cast<uintptr_t>(q) & 15) == 0; }

template <typename io_t, int K>
cudaError_t launch_vec(const ConvArgs& a, cudaStream_t s) {
    constexpr int U = 4;  // vectors per thread per pass
    const int64_t segs = a.rows * ((a.L / Vec<io_t>::V + 32 * U - 1) / (32 * U));
    auto kern = conv_vec_kernel<io_t, K, U>;
    // Up to 16 CTAs per SM, grid-striding beyond (MAMBA_CONV_BLOCKS=n: n per
    // SM).  Measured at [4, 4096, 4096] bf16: 16 per SM (four waves of the
    // four resident ones) 52.9 us, one resident wave 53.5 us, 8 per SM 53.3 us;
    // launched as a programmatic dependent 50.3 / 51.4 / 50.8 us.
    int dev = 0, sms = 148, per_sm = 16;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const char* nb = getenv("MAMBA_CONV_BLOCKS");
    if (nb && atoi(nb) > 0) per_sm = atoi(nb);
    const int64_t want = (segs + 7) / 8;  // 8 warps per block
    const int64_t cap = int64_t(sms) * per_sm;
    const unsigned grid = unsigned(want < 1 ? 1 : (want < cap ? want : cap));
    return launch_dependent(kern, dim3(grid), dim3(256), 0, s, "MAMBA_CONV_PDL", a);
}

template <typename io_t>
cudaError_t launch_conv_t(const ConvArgs& a, cudaStream_t s) {
    constexpr int V = Vec<io_t>::V;
    if (a.rows == 0) return cudaSuccess;
    if (a.L == 0) {
        if (!a.st_out || a.width == 1) return cudaSuccess;
        conv_state_copy_kernel<io_t><<<grid_for(a.rows * (a.width - 1), 256), 256, 0, s>>>(a);
        return cudaGetLastError();
    }
    const char* path = getenv("MAMBA_CONV_PATH");
    const bool force_scalar = path && path[0] == 's';
    const bool vec = !force_scalar && a.L % V == 0 && al16(a.x) && al16(a.out) &&
                     a.width - 1 <= V;
    if (vec) {
        switch (a.width) {
            case 1: return launch_vec<io_t, 1>(a, s);
            case 2: return launch_vec<io_t, 2>(a, s);
            case 3: return launch_vec<io_t, 3>(a, s);
            case 4: return launch_vec<io_t, 4>(a, s);
            case 5: return launch_vec<io_t, 5>(a, s);
            default:
                if constexpr (V >= 7) {
                    if (a.width == 6) return launch_vec<io_t, 6>(a, s);
                    if (a.width == 7) return launch_vec<io_t, 7>(a, s);
                    if (a.width == 8) return launch_vec<io_t, 8>(a, s);
                }
                break;
        }
    }
    conv_scalar_kernel<io_t><<<grid_for(a.rows * a.L, 256), 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_causal_conv1d(const void* x, const float* w, const float* bias,
                                 const void* st_in, void* out, void* st_out, int64_t batch,
                                 int64_t dim, int64_t L, int width, bool silu, bool bf16,
                                 cudaStream_t stream) {
    const ConvArgs a{x, w, bias, st_in, out, st_out, batch * dim, dim, L, width, silu};
    return bf16 ? launch_conv_t<__nv_bfloat16>(a, stream) : launch_conv_t<float>(a, stream);
}

cudaError_t launch_conv1d_update(void* state, const void* x, const float* w, const float* bias,
                                 void* out, int64_t batch, int64_t dim, int width, bool silu,
                                 bool bf16, cudaStream_t stream) {
    const int64_t rows = batch * dim;
    if (rows == 0) return cudaSuccess;
    const int grid = grid_for(rows, 256);
    if (bf16)
        conv_update_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(state, x, w, bias, out, rows,
                                                                     dim, width, silu);
    else
        conv_update_kernel<float><<<grid, 256, 0, stream>>>(state, x, w, bias, out, rows, dim,
                                                             width, silu);
    return cudaGetLastError();
}

}  // namespace mamba
