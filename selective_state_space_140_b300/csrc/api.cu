// C entry points of libmamba_scan.so: argument validation, then one launch.
// The declarations, layouts and error conventions are in include/mamba_scan.h.
#include <mutex>

#include "../../include/mamba_scan.h"
#include "../../include/mamba_scan_testing.h"
#include "common.cuh"
#include "scan_bwd.cuh"

namespace {

constexpr int64_t kMaxElems = int64_t(1) << 46;  // keeps every index far from overflow

size_t io_size(int io_dtype) { return io_dtype == MAMBA_BF16 ? 2 : 4; }

bool misaligned(const void* p, size_t align) {
    return p != nullptr && (reinterpret_cast<uintptr_t>(p) % align) != 0;
}

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

Range range_of(const void* p, int64_t elems, size_t esize) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return {lo, lo + uintptr_t(elems) * esize};
}

bool overlaps(Range a, Range b) {
    if (a.lo == 0 || b.lo == 0 || a.lo == a.hi || b.lo == b.hi) return false;
    return a.lo < b.hi && b.lo < a.hi;
}

bool size_ok(int64_t a, int64_t b, int64_t c) {
    if (a < 0 || b < 0 || c < 0) return false;
    if (a == 0 || b == 0 || c == 0) return true;
    if (a > kMaxElems / b) return false;
    return a * b <= kMaxElems / c;
}

// Scratch of mamba_selective_scan_fwd_noalloc: a fixed device buffer in this
// library's module (one copy per device), found once per device with
// cudaGetSymbolAddress.  A split needs at most about 256 * SMs * (dstate + 1)
// * 4 bytes (2.6 MB at dstate 16 on 148 SMs); 4 MiB covers that.
constexpr size_t kNoallocScratchBytes = size_t(4) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];  // set once the look-up on that device has succeeded

// Address of the fixed buffer on the current device.  Only a successful
// look-up is kept: a failed one (e.g. made while the module cannot be loaded)
// leaves no CUDA error behind and is retried by the next call.
cudaError_t noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess) {
            cudaGetLastError();
            return err;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

// Argument checks of the forward scan: MAMBA_OK to go on, else the status.
int check_scan_args(const void* u, const void* delta, const float* A_log, const void* B,
                    const void* C, const float* D, const void* z, const float* delta_bias,
                    void* y, float* last_state, int64_t batch, int64_t dim, int64_t seqlen,
                    int64_t dstate, int io_dtype) {
    if (io_dtype != MAMBA_F32 && io_dtype != MAMBA_BF16) return MAMBA_ERR_DTYPE;
    if (dstate < 1 || dstate > MAMBA_MAX_DSTATE) return MAMBA_ERR_DSTATE;
    if (!size_ok(batch, dim, seqlen) || !size_ok(batch, seqlen, dstate) ||
        !size_ok(batch, dim, dstate))
        return MAMBA_ERR_SIZE;
    // An array with no elements may be NULL (empty tensors have no storage).
    const bool has_elems = batch * dim * seqlen > 0, has_bc = batch * seqlen > 0;
    if ((has_elems && (!u || !delta || !y)) || (has_bc && (!B || !C)) || (dim > 0 && !A_log))
        return MAMBA_ERR_NULL;
    const size_t es = io_size(io_dtype);
    if (misaligned(u, es) || misaligned(delta, es) || misaligned(z, es) || misaligned(B, es) ||
        misaligned(C, es) || misaligned(y, es) || misaligned(A_log, 4) || misaligned(D, 4) ||
        misaligned(delta_bias, 4) || misaligned(last_state, 4))
        return MAMBA_ERR_ALIGN;
    const int64_t elems = batch * dim * seqlen;
    const Range ry = range_of(y, elems, es);
    const Range rs = last_state ? range_of(last_state, batch * dim * dstate, 4) : Range{0, 0};
    const Range ins[] = {range_of(u, elems, es), range_of(delta, elems, es),
                         z ? range_of(z, elems, es) : Range{0, 0},
                         range_of(B, batch * seqlen * dstate, es),
                         range_of(C, batch * seqlen * dstate, es),
                         range_of(A_log, dim * dstate, 4),
                         D ? range_of(D, dim, 4) : Range{0, 0},
                         delta_bias ? range_of(delta_bias, dim, 4) : Range{0, 0}};
    for (const Range& r : ins)
        if (overlaps(ry, r) || overlaps(rs, r)) return MAMBA_ERR_ALIAS;
    if (overlaps(ry, rs)) return MAMBA_ERR_ALIAS;
    return MAMBA_OK;
}

}  // namespace

extern "C" {

int mamba_abi_version(void) { return 1 * 10000 + 2 * 100 + 0; }

const char* mamba_status_string(int status) {
    switch (status) {
        case MAMBA_OK: return "MAMBA_OK";
        case MAMBA_ERR_NULL: return "MAMBA_ERR_NULL: a required pointer is NULL";
        case MAMBA_ERR_SIZE: return "MAMBA_ERR_SIZE: a size is negative or too large";
        case MAMBA_ERR_DSTATE: return "MAMBA_ERR_DSTATE: dstate must be in [1, 256]";
        case MAMBA_ERR_ALIGN: return "MAMBA_ERR_ALIGN: a pointer is not aligned to its element size";
        case MAMBA_ERR_DTYPE: return "MAMBA_ERR_DTYPE: io_dtype must be MAMBA_F32 or MAMBA_BF16";
        case MAMBA_ERR_LAUNCH: return "MAMBA_ERR_LAUNCH: the CUDA launch failed";
        case MAMBA_ERR_TIMEOUT: return "MAMBA_ERR_TIMEOUT: a bounded device-side wait gave up";
        case MAMBA_ERR_ALIAS: return "MAMBA_ERR_ALIAS: an output overlaps an input";
        case MAMBA_ERR_SCRATCH:
            return "MAMBA_ERR_SCRATCH: the split needs more than the 4 MiB fixed scratch of "
                   "mamba_selective_scan_fwd_noalloc";
        default: return "unknown mamba_status_t";
    }
}

int mamba_selective_scan_fwd(const void* u, const void* delta, const float* A_log, const void* B,
                             const void* C, const float* D, const void* z,
                             const float* delta_bias, int softplus_flag, void* y,
                             float* last_state, int64_t batch, int64_t dim, int64_t seqlen,
                             int64_t dstate, int io_dtype, mamba_stream_t stream) {
    const int st = check_scan_args(u, delta, A_log, B, C, D, z, delta_bias, y, last_state, batch,
                                   dim, seqlen, dstate, io_dtype);
    if (st != MAMBA_OK) return st;
    if (batch == 0 || dim == 0) return MAMBA_OK;

    mamba::ScanArgs a{u, delta, A_log, B, C, D, z, delta_bias, y, last_state,
                      batch, dim, seqlen, int(dstate), softplus_flag != 0};
    const mamba::ScanScratch scratch{nullptr, 0, true};
    const cudaError_t err = mamba::launch_scan_fwd(a, io_dtype == MAMBA_BF16,
                                                   reinterpret_cast<cudaStream_t>(stream), scratch);
    return err == cudaSuccess ? MAMBA_OK : MAMBA_ERR_LAUNCH;
}

int mamba_selective_scan_fwd_noalloc(const void* u, const void* delta, const float* A_log,
                                     const void* B, const void* C, const float* D,
                                     const void* z, const float* delta_bias, int softplus_flag,
                                     void* y, float* last_state, int64_t batch, int64_t dim,
                                     int64_t seqlen, int64_t dstate, int io_dtype,
                                     mamba_stream_t stream) {
    const int st = check_scan_args(u, delta, A_log, B, C, D, z, delta_bias, y, last_state, batch,
                                   dim, seqlen, dstate, io_dtype);
    if (st != MAMBA_OK) return st;
    if (batch == 0 || dim == 0) return MAMBA_OK;

    void* buf = nullptr;
    if (noalloc_scratch(&buf) != cudaSuccess) return MAMBA_ERR_LAUNCH;
    // Nothing in the buffer has to start at zero: the summary pass writes every
    // carried state and dt sum before the carry pass reads it.
    mamba::ScanArgs a{u, delta, A_log, B, C, D, z, delta_bias, y, last_state,
                      batch, dim, seqlen, int(dstate), softplus_flag != 0};
    const mamba::ScanScratch scratch{buf, kNoallocScratchBytes, false};
    const cudaError_t err = mamba::launch_scan_fwd(a, io_dtype == MAMBA_BF16,
                                                   reinterpret_cast<cudaStream_t>(stream), scratch);
    if (err == cudaErrorMemoryAllocation) return MAMBA_ERR_SCRATCH;
    return err == cudaSuccess ? MAMBA_OK : MAMBA_ERR_LAUNCH;
}

int mamba_selective_scan_fwd_ex(const void* u, const void* delta, const float* A_log,
                                const void* B, const void* C, const float* D, const void* z,
                                const float* delta_bias, int softplus_flag, const float* h0,
                                const unsigned char* reset, void* y, float* last_state,
                                int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                int io_dtype, mamba_stream_t stream) {
    const int st = check_scan_args(u, delta, A_log, B, C, D, z, delta_bias, y, last_state, batch,
                                   dim, seqlen, dstate, io_dtype);
    if (st != MAMBA_OK) return st;
    if (misaligned(h0, 4)) return MAMBA_ERR_ALIGN;
    // h0 may be last_state itself (continue a stream in place), but must not
    // otherwise overlap an output; the reset mask must not overlap one.
    const Range ry = range_of(y, batch * dim * seqlen, io_size(io_dtype));
    const Range rs = last_state ? range_of(last_state, batch * dim * dstate, 4) : Range{0, 0};
    const Range rh = h0 ? range_of(h0, batch * dim * dstate, 4) : Range{0, 0};
    const Range rr = reset ? range_of(reset, batch * seqlen, 1) : Range{0, 0};
    if (overlaps(rh, ry) || overlaps(rr, ry) || overlaps(rr, rs)) return MAMBA_ERR_ALIAS;
    if (overlaps(rh, rs) && static_cast<const void*>(h0) != static_cast<const void*>(last_state))
        return MAMBA_ERR_ALIAS;
    if (batch == 0 || dim == 0) return MAMBA_OK;

    mamba::ScanArgs a{u, delta, A_log, B, C, D, z, delta_bias, y, last_state,
                      batch, dim, seqlen, int(dstate), softplus_flag != 0, h0, reset};
    const mamba::ScanScratch scratch{nullptr, 0, true};
    const cudaError_t err = mamba::launch_scan_fwd(a, io_dtype == MAMBA_BF16,
                                                   reinterpret_cast<cudaStream_t>(stream), scratch);
    return err == cudaSuccess ? MAMBA_OK : MAMBA_ERR_LAUNCH;
}

int mamba_selective_scan_bwd(const void* u, const void* delta, const float* A_log, const void* B,
                             const void* C, const float* D, const void* z,
                             const float* delta_bias, int softplus_flag, const void* dout,
                             void* du, void* ddelta, void* dz, float* dA_log, float* dB,
                             float* dC, float* dD, float* ddelta_bias, int64_t batch,
                             int64_t dim, int64_t seqlen, int64_t dstate, int io_dtype,
                             mamba_stream_t stream) {
    return mamba_selective_scan_bwd_ex(u, delta, A_log, B, C, D, z, delta_bias, softplus_flag,
                                       nullptr, nullptr, dout, nullptr, du, ddelta, dz, dA_log,
                                       dB, dC, dD, ddelta_bias, nullptr, batch, dim, seqlen,
                                       dstate, io_dtype, stream);
}

int mamba_selective_scan_bwd_ex(const void* u, const void* delta, const float* A_log,
                                const void* B, const void* C, const float* D, const void* z,
                                const float* delta_bias, int softplus_flag, const float* h0,
                                const unsigned char* reset, const void* dout,
                                const float* dlast_state, void* du, void* ddelta, void* dz,
                                float* dA_log, float* dB, float* dC, float* dD,
                                float* ddelta_bias, float* dh0, int64_t batch,
                                int64_t dim, int64_t seqlen, int64_t dstate, int io_dtype,
                                mamba_stream_t stream) {
    if (io_dtype != MAMBA_F32 && io_dtype != MAMBA_BF16) return MAMBA_ERR_DTYPE;
    if (dstate < 1 || dstate > MAMBA_MAX_DSTATE) return MAMBA_ERR_DSTATE;
    if (!size_ok(batch, dim, seqlen) || !size_ok(batch, seqlen, dstate) ||
        !size_ok(batch, dim, dstate))
        return MAMBA_ERR_SIZE;
    const bool has_elems = batch * dim * seqlen > 0, has_bc = batch * seqlen > 0;
    if ((has_elems && (!u || !delta || !dout || !du || !ddelta || (z && !dz))) ||
        (has_bc && (!B || !C || !dB || !dC)) || (dim > 0 && (!A_log || !dA_log)))
        return MAMBA_ERR_NULL;
    const size_t es = io_size(io_dtype);
    if (misaligned(u, es) || misaligned(delta, es) || misaligned(z, es) || misaligned(B, es) ||
        misaligned(C, es) || misaligned(dout, es) || misaligned(du, es) ||
        misaligned(ddelta, es) || misaligned(dz, es) || misaligned(A_log, 4) ||
        misaligned(D, 4) || misaligned(delta_bias, 4) || misaligned(dA_log, 4) ||
        misaligned(dB, 4) || misaligned(dC, 4) || misaligned(dD, 4) ||
        misaligned(ddelta_bias, 4) || misaligned(h0, 4) || misaligned(dh0, 4) ||
        misaligned(dlast_state, 4))
        return MAMBA_ERR_ALIGN;
    const int64_t elems = batch * dim * seqlen, nbc = batch * seqlen * dstate;
    const int64_t nst = batch * dim * dstate;
    const Range ins[] = {range_of(u, elems, es), range_of(delta, elems, es),
                         z ? range_of(z, elems, es) : Range{0, 0}, range_of(B, nbc, es),
                         range_of(C, nbc, es), range_of(A_log, dim * dstate, 4),
                         D ? range_of(D, dim, 4) : Range{0, 0},
                         delta_bias ? range_of(delta_bias, dim, 4) : Range{0, 0},
                         range_of(dout, elems, es),
                         h0 ? range_of(h0, nst, 4) : Range{0, 0},
                         reset ? range_of(reset, batch * seqlen, 1) : Range{0, 0},
                         dlast_state ? range_of(dlast_state, nst, 4) : Range{0, 0}};
    const Range outs[] = {range_of(du, elems, es), range_of(ddelta, elems, es),
                          z ? range_of(dz, elems, es) : Range{0, 0},
                          range_of(dA_log, dim * dstate, 4), range_of(dB, nbc, 4),
                          range_of(dC, nbc, 4), dD ? range_of(dD, dim, 4) : Range{0, 0},
                          ddelta_bias ? range_of(ddelta_bias, dim, 4) : Range{0, 0},
                          dh0 ? range_of(dh0, nst, 4) : Range{0, 0}};
    for (size_t i = 0; i < sizeof(outs) / sizeof(outs[0]); ++i) {
        for (const Range& r : ins)
            if (overlaps(outs[i], r)) return MAMBA_ERR_ALIAS;
        for (size_t j = i + 1; j < sizeof(outs) / sizeof(outs[0]); ++j)
            if (overlaps(outs[i], outs[j])) return MAMBA_ERR_ALIAS;
    }
    if (dim == 0) return MAMBA_OK;

    mamba::ScanBwdArgs a{};
    a.f = mamba::ScanArgs{u, delta, A_log, B, C, D, z, delta_bias, nullptr, nullptr,
                          batch, dim, seqlen, int(dstate), softplus_flag != 0};
    a.f.h0 = h0;
    a.f.reset = reset;
    a.dout = dout;
    a.du = du;
    a.ddelta = ddelta;
    a.dz = z ? dz : nullptr;
    a.dA_log = dA_log;
    a.dB = dB;
    a.dC = dC;
    a.dD = dD;
    a.ddelta_bias = ddelta_bias;
    a.dlast = dlast_state;
    const cudaError_t err = mamba::launch_scan_bwd_ex(a, dh0, io_dtype == MAMBA_BF16,
                                                      reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? MAMBA_OK : MAMBA_ERR_LAUNCH;
}

int mamba_test_bounded_wait(int polls, mamba_stream_t stream) {
    if (polls < 1 || polls > (1 << 20)) return MAMBA_ERR_SIZE;
    const cudaError_t err =
        mamba::launch_bounded_wait_probe(uint32_t(polls), reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? MAMBA_OK : MAMBA_ERR_LAUNCH;
}

int mamba_device_status(mamba_stream_t stream) {
    unsigned int word = 0, dword = 0;
    const cudaError_t err =
        mamba::read_and_clear_device_error(&word, reinterpret_cast<cudaStream_t>(stream));
    if (err != cudaSuccess || mamba::read_and_clear_decode_error(&dword) != cudaSuccess)
        return MAMBA_ERR_LAUNCH;
    return ((word | dword) & mamba::kErrWaitTimeout) ? MAMBA_ERR_TIMEOUT : MAMBA_OK;
}

int mamba_selective_state_update(float* state, const void* x, const void* dt,
                                 const float* A_log, const void* B, const void* C,
                                 const float* D, const void* z, const float* dt_bias,
                                 int softplus_flag, void* out, int64_t batch, int64_t dim,
                                 int64_t dstate, int io_dtype, mamba_stream_t stream) {
    if (io_dtype != MAMBA_F32 && io_dtype != MAMBA_BF16) return MAMBA_ERR_DTYPE;
    if (dstate < 1 || dstate > MAMBA_MAX_DSTATE) return MAMBA_ERR_DSTATE;
    if (!size_ok(batch, dim, dstate)) return MAMBA_ERR_SIZE;
    if (batch * dim > 0 && (!state || !x || !dt || !out)) return MAMBA_ERR_NULL;
    if ((batch > 0 && (!B || !C)) || (dim > 0 && !A_log)) return MAMBA_ERR_NULL;
    const size_t es = io_size(io_dtype);
    if (misaligned(state, 4) || misaligned(x, es) || misaligned(dt, es) || misaligned(z, es) ||
        misaligned(B, es) || misaligned(C, es) || misaligned(out, es) || misaligned(A_log, 4) ||
        misaligned(D, 4) || misaligned(dt_bias, 4))
        return MAMBA_ERR_ALIGN;
    const Range ro = range_of(out, batch * dim, es);
    const Range rs = range_of(state, batch * dim * dstate, 4);
    const Range ins[] = {range_of(x, batch * dim, es), range_of(dt, batch * dim, es),
                         z ? range_of(z, batch * dim, es) : Range{0, 0},
                         range_of(B, batch * dstate, es), range_of(C, batch * dstate, es),
                         range_of(A_log, dim * dstate, 4),
                         D ? range_of(D, dim, 4) : Range{0, 0},
                         dt_bias ? range_of(dt_bias, dim, 4) : Range{0, 0}};
    for (const Range& r : ins)
        if (overlaps(ro, r) || overlaps(rs, r)) return MAMBA_ERR_ALIAS;
    if (overlaps(ro, rs)) return MAMBA_ERR_ALIAS;
    if (batch == 0 || dim == 0) return MAMBA_OK;

    mamba::StateUpdateArgs a{state, x, dt, A_log, B, C, D, z, dt_bias, out,
                             batch, dim, int(dstate), softplus_flag != 0};
    const cudaError_t err = mamba::launch_state_update(a, io_dtype == MAMBA_BF16,
                                                       reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? MAMBA_OK : MAMBA_ERR_LAUNCH;
}

int mamba_selective_scan_complex_fwd(const void* u, const void* delta, const float* A_log_re,
                                     const float* A_im, const void* B, const void* C,
                                     const float* D, const void* z, const float* delta_bias,
                                     int softplus_flag, void* y, float* last_state, int64_t batch,
                                     int64_t dim, int64_t seqlen, int64_t dstate, int io_dtype,
                                     mamba_stream_t stream) {
    if (io_dtype != MAMBA_F32 && io_dtype != MAMBA_BF16) return MAMBA_ERR_DTYPE;
    if (dstate < 1 || dstate > MAMBA_MAX_DSTATE) return MAMBA_ERR_DSTATE;
    if (!size_ok(batch, dim, seqlen) || !size_ok(batch, seqlen, 2 * dstate) ||
        !size_ok(batch, dim, 2 * dstate))
        return MAMBA_ERR_SIZE;
    const int64_t elems = batch * dim * seqlen, nbc = batch * seqlen * dstate * 2;
    const int64_t nst = batch * dim * dstate * 2;
    if ((elems > 0 && (!u || !delta || !y)) || (nbc > 0 && (!B || !C)) ||
        (dim > 0 && (!A_log_re || !A_im)))
        return MAMBA_ERR_NULL;
    const size_t es = io_size(io_dtype);
    if (misaligned(u, es) || misaligned(delta, es) || misaligned(z, es) || misaligned(B, es) ||
        misaligned(C, es) || misaligned(y, es) || misaligned(A_log_re, 4) ||
        misaligned(A_im, 4) || misaligned(D, 4) || misaligned(delta_bias, 4) ||
        misaligned(last_state, 8))
        return MAMBA_ERR_ALIGN;
    const Range ry = range_of(y, elems, es);
    const Range rh = last_state ? range_of(last_state, nst, 4) : Range{0, 0};
    const Range ins[] = {range_of(u, elems, es), range_of(delta, elems, es),
                         z ? range_of(z, elems, es) : Range{0, 0}, range_of(B, nbc, es),
                         range_of(C, nbc, es), range_of(A_log_re, dim * dstate, 4),
                         range_of(A_im, dim * dstate, 4), D ? range_of(D, dim, 4) : Range{0, 0},
                         delta_bias ? range_of(delta_bias, dim, 4) : Range{0, 0}};
    for (const Range& r : ins)
        if (overlaps(ry, r) || overlaps(rh, r)) return MAMBA_ERR_ALIAS;
    if (overlaps(ry, rh)) return MAMBA_ERR_ALIAS;
    if (batch == 0 || dim == 0) return MAMBA_OK;
    const cudaError_t err = mamba::launch_scan_complex(
        u, delta, A_log_re, A_im, B, C, D, z, delta_bias, softplus_flag != 0, y, last_state,
        batch, dim, seqlen, int(dstate), io_dtype == MAMBA_BF16,
        reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? MAMBA_OK : MAMBA_ERR_LAUNCH;
}

int mamba_causal_conv1d_fwd(const void* x, const float* weight, const float* bias,
                            const void* initial_state, int silu_flag, void* out,
                            void* final_state, int64_t batch, int64_t dim, int64_t seqlen,
                            int64_t width, int io_dtype, mamba_stream_t stream) {
    if (io_dtype != MAMBA_F32 && io_dtype != MAMBA_BF16) return MAMBA_ERR_DTYPE;
    if (width < 1 || width > MAMBA_MAX_CONV_WIDTH) return MAMBA_ERR_SIZE;
    if (!size_ok(batch, dim, seqlen) || !size_ok(batch, dim, width)) return MAMBA_ERR_SIZE;
    const int64_t elems = batch * dim * seqlen, nst = batch * dim * (width - 1);
    if ((elems > 0 && (!x || !out)) || (dim > 0 && !weight)) return MAMBA_ERR_NULL;
    const size_t es = io_size(io_dtype);
    if (misaligned(x, es) || misaligned(out, es) || misaligned(initial_state, es) ||
        misaligned(final_state, es) || misaligned(weight, 4) || misaligned(bias, 4))
        return MAMBA_ERR_ALIGN;
    const Range ro = range_of(out, elems, es);
    const Range rf = final_state ? range_of(final_state, nst, es) : Range{0, 0};
    const Range ins[] = {range_of(x, elems, es), range_of(weight, dim * width, 4),
                         bias ? range_of(bias, dim, 4) : Range{0, 0},
                         initial_state ? range_of(initial_state, nst, es) : Range{0, 0}};
    for (const Range& r : ins)
        if (overlaps(ro, r) || overlaps(rf, r)) return MAMBA_ERR_ALIAS;
    if (overlaps(ro, rf)) return MAMBA_ERR_ALIAS;
    if (batch == 0 || dim == 0) return MAMBA_OK;
    const cudaError_t err = mamba::launch_causal_conv1d(
        x, weight, bias, initial_state, out, final_state, batch, dim, seqlen, int(width),
        silu_flag != 0, io_dtype == MAMBA_BF16, reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? MAMBA_OK : MAMBA_ERR_LAUNCH;
}

int mamba_causal_conv1d_update(void* conv_state, const void* x, const float* weight,
                               const float* bias, int silu_flag, void* out, int64_t batch,
                               int64_t dim, int64_t width, int io_dtype, mamba_stream_t stream) {
    if (io_dtype != MAMBA_F32 && io_dtype != MAMBA_BF16) return MAMBA_ERR_DTYPE;
    if (width < 1 || width > MAMBA_MAX_CONV_WIDTH) return MAMBA_ERR_SIZE;
    if (!size_ok(batch, dim, width)) return MAMBA_ERR_SIZE;
    const int64_t rows = batch * dim, nst = rows * (width - 1);
    if ((rows > 0 && (!x || !out || (width > 1 && !conv_state))) || (dim > 0 && !weight))
        return MAMBA_ERR_NULL;
    const size_t es = io_size(io_dtype);
    if (misaligned(conv_state, es) || misaligned(x, es) || misaligned(out, es) ||
        misaligned(weight, 4) || misaligned(bias, 4))
        return MAMBA_ERR_ALIGN;
    const Range ro = range_of(out, rows, es);
    const Range rs = width > 1 ? range_of(conv_state, nst, es) : Range{0, 0};
    const Range ins[] = {range_of(x, rows, es), range_of(weight, dim * width, 4),
                         bias ? range_of(bias, dim, 4) : Range{0, 0}};
    for (const Range& r : ins)
        if (overlaps(ro, r) || overlaps(rs, r)) return MAMBA_ERR_ALIAS;
    if (overlaps(ro, rs)) return MAMBA_ERR_ALIAS;
    if (rows == 0) return MAMBA_OK;
    const cudaError_t err = mamba::launch_conv1d_update(
        conv_state, x, weight, bias, out, batch, dim, int(width), silu_flag != 0,
        io_dtype == MAMBA_BF16, reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? MAMBA_OK : MAMBA_ERR_LAUNCH;
}

}  // extern "C"
