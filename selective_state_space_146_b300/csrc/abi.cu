// abi.cu -- the C ABI (include/ssscan.h): argument checks on the host, then
// dispatch to the kernels on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ssscan.h"

namespace ss {

// ---------------------------------------------------------------------------
// Per-device state: the device error word and the SM count.

__device__ unsigned g_device_error;

constexpr int kMaxDevices = 64;
static unsigned* g_err_ptr[kMaxDevices];
static int g_sms[kMaxDevices];
static std::mutex g_mu;
static std::atomic<uint64_t> g_launches{0};

void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

static int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

static unsigned* device_error_ptr() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<unsigned*>(p);
    }
    return g_err_ptr[dev];
}

int sm_count_current() {
    const int dev = current_device();
    if (dev < 0) return 148;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sms[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        g_sms[dev] = v > 0 ? v : 148;
    }
    return g_sms[dev];
}

void* tensor_map_encoder() {
    static void* fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = f;
    });
    return fn;
}

// Diagnostic switches (ss_debug_set_path): -1 is the library's own choice.
static std::atomic<int> g_debug[SS_DEBUG_COUNT] = {-1, -1, -1, -1, -1, -1, -1, -1, -1, -1};
static_assert(SS_DEBUG_COUNT == 10, "one initial -1 per switch");

int debug_path(int which) {
    return which >= 0 && which < SS_DEBUG_COUNT ? g_debug[which].load(std::memory_order_relaxed) : -1;
}

// SS_DEBUG_FAULT_ALLOC = 1 makes every stream-ordered scratch allocation
// report failure (a host-side fault injection for the tests of SS_ERR_ALLOC).
static bool fault_alloc() { return debug_path(SS_DEBUG_FAULT_ALLOC) == 1; }

static void* scratch_alloc_async(size_t bytes, cudaStream_t st, void*) {
    if (fault_alloc()) return nullptr;
    void* p = nullptr;
    if (cudaMallocAsync(&p, bytes, st) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return p;
}

static void scratch_free_async(void* p, cudaStream_t st, void*) { cudaFreeAsync(p, st); }

// ---------------------------------------------------------------------------
// Argument checks.

static int elem_size(int dtype) { return dtype == SS_BF16 ? 2 : dtype == SS_F32 ? 4 : 0; }

static int check_tensor(const ss_tensor* t, int ndim) {
    if (!t) return SS_ERR_INVALID_ARG;
    if (t->ndim != ndim) return SS_ERR_SHAPE;
    int64_t numel = 1;
    for (int i = 0; i < ndim; ++i) {
        if (t->shape[i] < 0 || t->stride[i] < 0) return SS_ERR_SHAPE;
        numel *= t->shape[i];
    }
    if (!elem_size(t->dtype)) return SS_ERR_DTYPE;
    if (numel > 0) {
        if (!t->data) return SS_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(t->data) % elem_size(t->dtype)) return SS_ERR_ALIGNMENT;
    }
    return SS_OK;
}

static bool same_shape(const ss_tensor* a, const ss_tensor* b) {
    if (a->ndim != b->ndim) return false;
    for (int i = 0; i < a->ndim; ++i)
        if (a->shape[i] != b->shape[i]) return false;
    return true;
}

#define SS_TRY(expr)                 \
    do {                             \
        int _rc = (expr);            \
        if (_rc != SS_OK) return _rc; \
    } while (0)

// ---------------------------------------------------------------------------
// Fixed scratch for ss_selective_scan_fwd_noalloc.
//
// The segment summaries of the selective scan come from this array instead of
// cudaMallocAsync.  It is a file-scope device array, so every GPU that loads
// the library holds it until the process exits.  In host code its name is
// only a stand-in: the device address is taken once per device with
// cudaGetSymbolAddress (first call on that device, with the device current)
// and passed to the kernels as a plain pointer.
constexpr size_t kFixedScratchBytes = size_t(4) << 20;  // 4 MiB per device
static __device__ __align__(256) unsigned char g_fixed_scratch[kFixedScratchBytes];
static void* g_fixed_scratch_ptr[kMaxDevices];

static void* fixed_scratch_address() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_fixed_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fixed_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return nullptr;
        }
        g_fixed_scratch_ptr[dev] = p;
    }
    return g_fixed_scratch_ptr[dev];
}

struct FixedScratch {
    void* base;
    bool too_large;  // a request exceeded kFixedScratchBytes
};

static void* fixed_scratch_alloc(size_t bytes, cudaStream_t, void* ctx) {
    auto* fs = static_cast<FixedScratch*>(ctx);
    if (bytes > kFixedScratchBytes) {
        fs->too_large = true;
        return nullptr;
    }
    return fs->base;
}

static void fixed_scratch_release(void*, cudaStream_t, void*) {}

}  // namespace ss

using namespace ss;

extern "C" {

// Checks and ScanArgs assembly shared by the scans with and without an
// initial state.
static int selective_args(const ss_tensor* u, const ss_tensor* delta, const ss_tensor* A,
                          const ss_tensor* B, const ss_tensor* C, const ss_tensor* D,
                          const ss_tensor* z, const ss_tensor* delta_bias, int softplus,
                          const ss_tensor* h0, ss_tensor* y, ss_tensor* last_state,
                          ScanArgs* out, bool* nothing_to_do) {
    *nothing_to_do = false;
    SS_TRY(check_tensor(u, 3));
    SS_TRY(check_tensor(delta, 3));
    SS_TRY(check_tensor(A, 2));
    // B, C: (Bsz, N, L), or (Bsz, G, N, L) with one B, C per group of channels
    if (!B || !C) return SS_ERR_INVALID_ARG;
    const bool grouped = B->ndim == 4;
    SS_TRY(check_tensor(B, grouped ? 4 : 3));
    SS_TRY(check_tensor(C, grouped ? 4 : 3));
    SS_TRY(check_tensor(y, 3));
    if (D) SS_TRY(check_tensor(D, 1));
    if (z) SS_TRY(check_tensor(z, 3));
    if (delta_bias) SS_TRY(check_tensor(delta_bias, 1));
    if (last_state) SS_TRY(check_tensor(last_state, 3));
    if (h0) SS_TRY(check_tensor(h0, 3));
    if (softplus != 0 && softplus != 1) return SS_ERR_INVALID_ARG;

    const int dt = u->dtype;
    if (delta->dtype != dt || B->dtype != dt || C->dtype != dt || y->dtype != dt ||
        (z && z->dtype != dt))
        return SS_ERR_DTYPE;
    if (A->dtype != SS_F32 || (D && D->dtype != SS_F32) ||
        (delta_bias && delta_bias->dtype != SS_F32) || (last_state && last_state->dtype != SS_F32) ||
        (h0 && h0->dtype != SS_F32))
        return SS_ERR_DTYPE;

    const int64_t Bsz = u->shape[0], Dch = u->shape[1], L = u->shape[2], N = A->shape[1];
    if (!same_shape(delta, u) || !same_shape(y, u) || (z && !same_shape(z, u)))
        return SS_ERR_SHAPE;
    if (A->shape[0] != Dch) return SS_ERR_SHAPE;
    const int nd = grouped ? 1 : 0;  // index shift of the (N, L) dims
    const int64_t G = grouped ? B->shape[1] : 1;
    if (B->shape[0] != Bsz || B->shape[1 + nd] != N || B->shape[2 + nd] != L) return SS_ERR_SHAPE;
    if (!same_shape(C, B)) return SS_ERR_SHAPE;
    if (G < 1 || (Dch > 0 && Dch % G != 0)) return SS_ERR_SHAPE;
    if (D && D->shape[0] != Dch) return SS_ERR_SHAPE;
    if (delta_bias && delta_bias->shape[0] != Dch) return SS_ERR_SHAPE;
    if (last_state && (last_state->shape[0] != Bsz || last_state->shape[1] != Dch ||
                       last_state->shape[2] != N))
        return SS_ERR_SHAPE;
    if (h0 && (h0->shape[0] != Bsz || h0->shape[1] != Dch || h0->shape[2] != N)) return SS_ERR_SHAPE;
    if (N < 1) return SS_ERR_SHAPE;
    if (N > 256) return SS_ERR_UNSUPPORTED;
    if (Bsz * Dch >= (int64_t(1) << 31) || L >= (int64_t(1) << 31)) return SS_ERR_UNSUPPORTED;
    if (Bsz == 0 || Dch == 0 || (L == 0 && !last_state)) {
        *nothing_to_do = true;
        return SS_OK;
    }

    ScanArgs a{};
    a.Bsz = (int)Bsz; a.D = (int)Dch; a.N = (int)N; a.L = (int)L; a.dtype = dt;
    a.u = u->data; a.su_b = u->stride[0]; a.su_d = u->stride[1]; a.su_t = u->stride[2];
    a.dl = delta->data; a.sdl_b = delta->stride[0]; a.sdl_d = delta->stride[1]; a.sdl_t = delta->stride[2];
    if (z) { a.z = z->data; a.sz_b = z->stride[0]; a.sz_d = z->stride[1]; a.sz_t = z->stride[2]; }
    a.y = y->data; a.sy_b = y->stride[0]; a.sy_d = y->stride[1]; a.sy_t = y->stride[2];
    a.Bm = B->data; a.sB_b = B->stride[0];
    a.sB_n = B->stride[1 + nd]; a.sB_t = B->stride[2 + nd];
    a.Cm = C->data; a.sC_b = C->stride[0];
    a.sC_n = C->stride[1 + nd]; a.sC_t = C->stride[2 + nd];
    a.G = (int)G;
    a.sB_g = grouped ? B->stride[1] : 0;
    a.sC_g = grouped ? C->stride[1] : 0;
    a.A = static_cast<const float*>(A->data); a.sA_d = A->stride[0]; a.sA_n = A->stride[1];
    if (D) { a.Dv = static_cast<const float*>(D->data); a.sD = D->stride[0]; }
    if (delta_bias) { a.bias = static_cast<const float*>(delta_bias->data); a.sbias = delta_bias->stride[0]; }
    if (last_state) {
        a.last = static_cast<float*>(last_state->data);
        a.sl_b = last_state->stride[0]; a.sl_d = last_state->stride[1]; a.sl_n = last_state->stride[2];
    }
    if (h0) {
        a.h0 = static_cast<const float*>(h0->data);
        a.sh_b = h0->stride[0]; a.sh_d = h0->stride[1]; a.sh_n = h0->stride[2];
    }
    a.softplus = softplus;
    *out = a;
    return SS_OK;
}

int ss_selective_scan_fwd_init(const ss_tensor* u, const ss_tensor* delta, const ss_tensor* A,
                               const ss_tensor* B, const ss_tensor* C, const ss_tensor* D,
                               const ss_tensor* z, const ss_tensor* delta_bias, int softplus,
                               const ss_tensor* initial_state, ss_tensor* y,
                               ss_tensor* last_state, void* stream) {
    ScanArgs a{};
    bool nothing = false;
    SS_TRY(selective_args(u, delta, A, B, C, D, z, delta_bias, softplus, initial_state, y,
                          last_state, &a, &nothing));
    if (nothing) return SS_OK;
    a.err = device_error_ptr();
    if (!a.err) return SS_ERR_CUDA;
    Scratch sc{scratch_alloc_async, scratch_free_async, nullptr};
    return launch_selective(a, static_cast<cudaStream_t>(stream), sc);
}

int ss_conv_selective_scan_fwd(const ss_tensor* x, const ss_tensor* conv_weight,
                               const ss_tensor* conv_bias, const ss_tensor* delta,
                               const ss_tensor* A, const ss_tensor* B, const ss_tensor* C,
                               const ss_tensor* D, const ss_tensor* z,
                               const ss_tensor* delta_bias, int softplus, ss_tensor* y,
                               ss_tensor* last_state, void* stream) {
    SS_TRY(check_tensor(conv_weight, 2));
    if (conv_bias) SS_TRY(check_tensor(conv_bias, 1));
    if (conv_weight->dtype != SS_F32 || (conv_bias && conv_bias->dtype != SS_F32))
        return SS_ERR_DTYPE;
    ScanArgs a{};
    bool nothing = false;
    SS_TRY(selective_args(x, delta, A, B, C, D, z, delta_bias, softplus, nullptr, y, last_state,
                          &a, &nothing));
    const int64_t W = conv_weight->shape[1];
    if (conv_weight->shape[0] != x->shape[1] || (conv_bias && conv_bias->shape[0] != x->shape[1]))
        return SS_ERR_SHAPE;
    if (W < 1) return SS_ERR_SHAPE;
    if (W > 4) return SS_ERR_UNSUPPORTED;
    if (nothing) return SS_OK;
    a.cw = static_cast<const float*>(conv_weight->data);
    a.scw_d = conv_weight->stride[0]; a.scw_k = conv_weight->stride[1];
    if (conv_bias) { a.cb = static_cast<const float*>(conv_bias->data); a.scb = conv_bias->stride[0]; }
    a.cwidth = (int)W;
    a.err = device_error_ptr();
    if (!a.err) return SS_ERR_CUDA;
    Scratch sc{scratch_alloc_async, scratch_free_async, nullptr};
    return launch_selective(a, static_cast<cudaStream_t>(stream), sc);
}

int ss_debug_set_path(int which, int value) {
    if (which < 0 || which >= SS_DEBUG_COUNT) return SS_ERR_INVALID_ARG;
    g_debug[which].store(value < 0 ? -1 : value, std::memory_order_relaxed);
    return SS_OK;
}

int ss_selective_scan_fwd(const ss_tensor* u, const ss_tensor* delta, const ss_tensor* A,
                          const ss_tensor* B, const ss_tensor* C, const ss_tensor* D,
                          const ss_tensor* z, const ss_tensor* delta_bias, int softplus,
                          ss_tensor* y, ss_tensor* last_state, void* stream) {
    return ss_selective_scan_fwd_init(u, delta, A, B, C, D, z, delta_bias, softplus, nullptr, y,
                                      last_state, stream);
}

static bool is_contiguous(const ss_tensor* t);

// The checkpoint tensor of the forward-for-training / backward pair: fp32,
// (batch, channels, ceil(L / 8), 16), contiguous, 16-byte aligned.
static int check_ckpt(const ss_tensor* ck, const ss_tensor* u) {
    SS_TRY(check_tensor(ck, 4));
    if (ck->dtype != SS_F32) return SS_ERR_DTYPE;
    const int64_t L = u->shape[2];
    if (ck->shape[0] != u->shape[0] || ck->shape[1] != u->shape[1] || ck->shape[2] != (L + 7) / 8 ||
        ck->shape[3] != 16)
        return SS_ERR_SHAPE;
    if (!is_contiguous(ck)) return SS_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(ck->data) % 16) return SS_ERR_ALIGNMENT;
    return SS_OK;
}

int ss_selective_scan_fwd_ckpt(const ss_tensor* u, const ss_tensor* delta, const ss_tensor* A,
                               const ss_tensor* B, const ss_tensor* C, const ss_tensor* D,
                               const ss_tensor* z, const ss_tensor* delta_bias, int softplus,
                               ss_tensor* y, ss_tensor* last_state, ss_tensor* ckpt,
                               void* stream) {
    ScanArgs a{};
    bool nothing = false;
    if (B && B->ndim == 4) return SS_ERR_UNSUPPORTED;  // B, C shared per batch row only
    SS_TRY(selective_args(u, delta, A, B, C, D, z, delta_bias, softplus, nullptr, y, last_state,
                          &a, &nothing));
    SS_TRY(check_ckpt(ckpt, u));
    if (nothing) return SS_OK;
    a.ckpt = static_cast<float*>(ckpt->data);
    a.err = device_error_ptr();
    if (!a.err) return SS_ERR_CUDA;
    Scratch sc{scratch_alloc_async, scratch_free_async, nullptr};
    return launch_selective(a, static_cast<cudaStream_t>(stream), sc);
}

int ss_selective_scan_fwd_noalloc(const ss_tensor* u, const ss_tensor* delta, const ss_tensor* A,
                                  const ss_tensor* B, const ss_tensor* C, const ss_tensor* D,
                                  const ss_tensor* z, const ss_tensor* delta_bias, int softplus,
                                  ss_tensor* y, ss_tensor* last_state, void* stream) {
    ScanArgs a{};
    bool nothing = false;
    SS_TRY(selective_args(u, delta, A, B, C, D, z, delta_bias, softplus, nullptr, y, last_state,
                          &a, &nothing));
    if (nothing) return SS_OK;
    a.err = device_error_ptr();
    if (!a.err) return SS_ERR_CUDA;
    FixedScratch fs{fixed_scratch_address(), false};
    if (!fs.base) return SS_ERR_CUDA;
    Scratch sc{fixed_scratch_alloc, fixed_scratch_release, &fs, kFixedScratchBytes};
    const int rc = launch_selective(a, static_cast<cudaStream_t>(stream), sc);
    // the summaries would not fit the fixed buffer: nothing was launched
    if (rc == SS_ERR_ALLOC && fs.too_large) return SS_ERR_UNSUPPORTED;
    return rc;
}

static bool is_contiguous(const ss_tensor* t) {
    for (int i = 0; i < t->ndim; ++i)
        if (t->shape[i] == 0) return true;  // empty: nothing is addressed
    int64_t expect = 1;
    for (int i = t->ndim - 1; i >= 0; --i) {
        if (t->shape[i] != 1 && t->stride[i] != expect) return false;
        expect *= t->shape[i];
    }
    return true;
}

// An fp32 gradient output: the given shape, contiguous.
static int check_grad_f32(const ss_tensor* t, int ndim, const int64_t* shape) {
    SS_TRY(check_tensor(t, ndim));
    if (t->dtype != SS_F32) return SS_ERR_DTYPE;
    for (int i = 0; i < ndim; ++i)
        if (t->shape[i] != shape[i]) return SS_ERR_SHAPE;
    if (!is_contiguous(t)) return SS_ERR_UNSUPPORTED;
    return SS_OK;
}

static int selective_bwd(const ss_tensor* u, const ss_tensor* delta, const ss_tensor* A,
                         const ss_tensor* B, const ss_tensor* C, const ss_tensor* D,
                         const ss_tensor* z, const ss_tensor* delta_bias, int softplus,
                         const ss_tensor* dout, const ss_tensor* ckpt, ss_tensor* du,
                         ss_tensor* ddelta, ss_tensor* dA, ss_tensor* dB, ss_tensor* dC,
                         ss_tensor* dD, ss_tensor* dz, ss_tensor* ddelta_bias, void* stream) {
    ScanArgs f{};
    bool nothing = false;
    if (B && B->ndim == 4) return SS_ERR_UNSUPPORTED;  // B, C shared per batch row only
    // the forward inputs are checked as for the forward scan, dout in the place of y
    SS_TRY(selective_args(u, delta, A, B, C, D, z, delta_bias, softplus, nullptr,
                          const_cast<ss_tensor*>(dout), nullptr, &f, &nothing));
    SS_TRY(check_tensor(du, 3));
    SS_TRY(check_tensor(ddelta, 3));
    if (!same_shape(du, u) || !same_shape(ddelta, u)) return SS_ERR_SHAPE;
    if (du->dtype != u->dtype || ddelta->dtype != u->dtype) return SS_ERR_DTYPE;
    if (!z != !dz || !D != !dD || !delta_bias != !ddelta_bias) return SS_ERR_INVALID_ARG;
    if (dz) {
        SS_TRY(check_tensor(dz, 3));
        if (!same_shape(dz, u)) return SS_ERR_SHAPE;
        if (dz->dtype != u->dtype) return SS_ERR_DTYPE;
    }
    const int64_t Bsz = u->shape[0], Dch = u->shape[1], L = u->shape[2], N = A->shape[1];
    const int64_t sDN[2] = {Dch, N}, sBNL[3] = {Bsz, N, L}, sD1[1] = {Dch};
    SS_TRY(check_grad_f32(dA, 2, sDN));
    SS_TRY(check_grad_f32(dB, 3, sBNL));
    SS_TRY(check_grad_f32(dC, 3, sBNL));
    if (dD) SS_TRY(check_grad_f32(dD, 1, sD1));
    if (ddelta_bias) SS_TRY(check_grad_f32(ddelta_bias, 1, sD1));
    if (N > 16) return SS_ERR_UNSUPPORTED;
    if (ckpt) SS_TRY(check_ckpt(ckpt, u));

    BwdArgs a{};
    a.Bsz = (int)Bsz; a.D = (int)Dch; a.N = (int)N; a.L = (int)L; a.dtype = u->dtype;
    a.dA = static_cast<float*>(dA->data);
    a.dB = static_cast<float*>(dB->data);
    a.dC = static_cast<float*>(dC->data);
    a.dD = dD ? static_cast<float*>(dD->data) : nullptr;
    a.dbias = ddelta_bias ? static_cast<float*>(ddelta_bias->data) : nullptr;
    if (!nothing) {  // else the launcher only zeroes the sums
        a.u = f.u; a.su_b = f.su_b; a.su_d = f.su_d; a.su_t = f.su_t;
        a.dl = f.dl; a.sdl_b = f.sdl_b; a.sdl_d = f.sdl_d; a.sdl_t = f.sdl_t;
        a.z = f.z; a.sz_b = f.sz_b; a.sz_d = f.sz_d; a.sz_t = f.sz_t;
        a.dout = f.y; a.sg_b = f.sy_b; a.sg_d = f.sy_d; a.sg_t = f.sy_t;
        a.Bm = f.Bm; a.sB_b = f.sB_b; a.sB_n = f.sB_n; a.sB_t = f.sB_t;
        a.Cm = f.Cm; a.sC_b = f.sC_b; a.sC_n = f.sC_n; a.sC_t = f.sC_t;
        a.A = f.A; a.sA_d = f.sA_d; a.sA_n = f.sA_n;
        a.Dv = f.Dv; a.sD = f.sD;
        a.bias = f.bias; a.sbias = f.sbias;
        a.softplus = softplus;
        a.du = du->data; a.sdu_b = du->stride[0]; a.sdu_d = du->stride[1]; a.sdu_t = du->stride[2];
        a.ddl = ddelta->data;
        a.sddl_b = ddelta->stride[0]; a.sddl_d = ddelta->stride[1]; a.sddl_t = ddelta->stride[2];
        if (dz) { a.dz = dz->data; a.sdz_b = dz->stride[0]; a.sdz_d = dz->stride[1]; a.sdz_t = dz->stride[2]; }
    }
    a.ckpt_in = ckpt ? static_cast<const float*>(ckpt->data) : nullptr;
    a.err = device_error_ptr();
    if (!a.err) return SS_ERR_CUDA;
    Scratch sc{scratch_alloc_async, scratch_free_async, nullptr};
    return launch_selective_bwd(a, static_cast<cudaStream_t>(stream), sc);
}

int ss_selective_scan_bwd(const ss_tensor* u, const ss_tensor* delta, const ss_tensor* A,
                          const ss_tensor* B, const ss_tensor* C, const ss_tensor* D,
                          const ss_tensor* z, const ss_tensor* delta_bias, int softplus,
                          const ss_tensor* dout, ss_tensor* du, ss_tensor* ddelta, ss_tensor* dA,
                          ss_tensor* dB, ss_tensor* dC, ss_tensor* dD, ss_tensor* dz,
                          ss_tensor* ddelta_bias, void* stream) {
    return selective_bwd(u, delta, A, B, C, D, z, delta_bias, softplus, dout, nullptr, du, ddelta,
                         dA, dB, dC, dD, dz, ddelta_bias, stream);
}

int ss_selective_scan_bwd_ckpt(const ss_tensor* u, const ss_tensor* delta, const ss_tensor* A,
                               const ss_tensor* B, const ss_tensor* C, const ss_tensor* D,
                               const ss_tensor* z, const ss_tensor* delta_bias, int softplus,
                               const ss_tensor* dout, const ss_tensor* ckpt, ss_tensor* du,
                               ss_tensor* ddelta, ss_tensor* dA, ss_tensor* dB, ss_tensor* dC,
                               ss_tensor* dD, ss_tensor* dz, ss_tensor* ddelta_bias, void* stream) {
    if (!ckpt) return SS_ERR_INVALID_ARG;
    return selective_bwd(u, delta, A, B, C, D, z, delta_bias, softplus, dout, ckpt, du, ddelta,
                         dA, dB, dC, dD, dz, ddelta_bias, stream);
}

// ---------------------------------------------------------------------------
// Host buffers in and out: ss_selective_scan_fwd_host.  The batch is cut into
// chunks of rows, or of one row's channels when a row is large; chunks
// alternate between the caller's stream and one side stream per device, so the
// copy in of one chunk overlaps the scan of the one before and the copy out of
// the one before that.

static cudaStream_t g_side[kMaxDevices];

static cudaStream_t side_stream() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_side[dev]) {
        cudaStream_t s = nullptr;
        if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_side[dev] = s;
    }
    return g_side[dev];
}

static size_t numel(const ss_tensor* t) {
    size_t n = 1;
    for (int i = 0; i < t->ndim; ++i) n *= (size_t)t->shape[i];
    return n;
}

static size_t round256(size_t n) { return (n + 255) & ~size_t(255); }

int ss_selective_scan_fwd_host(const ss_tensor* u, const ss_tensor* delta, const ss_tensor* A,
                               const ss_tensor* B, const ss_tensor* C, const ss_tensor* D,
                               const ss_tensor* z, const ss_tensor* delta_bias, int softplus,
                               ss_tensor* y, ss_tensor* last_state, void* stream) {
    ScanArgs a{};
    bool nothing = false;
    SS_TRY(selective_args(u, delta, A, B, C, D, z, delta_bias, softplus, nullptr, y, last_state,
                          &a, &nothing));
    if (nothing) return SS_OK;
    for (const ss_tensor* t : {u, delta, A, B, C, D, z, delta_bias, static_cast<const ss_tensor*>(y),
                               static_cast<const ss_tensor*>(last_state)})
        if (t && !is_contiguous(t)) return SS_ERR_UNSUPPORTED;
    a.err = device_error_ptr();
    if (!a.err) return SS_ERR_CUDA;
    cudaStream_t s0 = static_cast<cudaStream_t>(stream);
    cudaStream_t s1 = side_stream();
    if (!s1) return SS_ERR_CUDA;

    const int es = elem_size(u->dtype);
    const int64_t Bsz = a.Bsz, Dch = a.D, L = a.L, N = a.N, G = a.G > 1 ? a.G : 1;
    const size_t act_ch = (size_t)L * es;               // one channel of u / delta / z / y
    const size_t act_row = (size_t)Dch * act_ch;        // one batch row of them
    const size_t bc_row = (size_t)G * N * L * es;       // one batch row of B or C
    const size_t st_ch = (size_t)N * sizeof(float);
    const size_t in_row = act_row * (z ? 3 : 2) + 2 * bc_row;
    // Chunks of about 32 MB of inputs: whole batch rows while a row is
    // smaller (at least two chunks when there are two rows), else blocks of
    // channels of one row (whole channel groups when B, C are grouped), so
    // that even one long row overlaps its copies with the scan.
    constexpr size_t kChunkBytes = size_t(32) << 20;
    int64_t rows = 1, cd = Dch;
    if (in_row <= kChunkBytes) {
        rows = std::max<int64_t>(1, (int64_t)(kChunkBytes / std::max<size_t>(in_row, 1)));
        if (Bsz >= 2) rows = std::min<int64_t>(rows, (Bsz + 1) / 2);
        rows = std::min<int64_t>(rows, Bsz);
    } else {
        const int64_t gsz = Dch / G;  // channels per group (all of them when shared)
        const int64_t unit = G > 1 ? gsz : 1;
        cd = (int64_t)(kChunkBytes / (act_ch * (z ? 3 : 2)));
        cd = std::max<int64_t>(unit, cd / unit * unit);
        cd = std::min<int64_t>(cd, Dch);
    }
    const int64_t cblocks = (Dch + cd - 1) / cd;  // channel blocks per batch row
    const int64_t nchunk = cd < Dch ? Bsz * cblocks : (Bsz + rows - 1) / rows;
    const int nset = nchunk > 1 ? 2 : 1;

    // device layout: A, D, bias once; then `nset` sets of chunk buffers
    const size_t szA = round256(numel(A) * sizeof(float));
    const size_t szD = D ? round256(Dch * sizeof(float)) : 0;
    const size_t szb = delta_bias ? round256(Dch * sizeof(float)) : 0;
    const size_t cact = round256(act_ch * cd * rows), cbc = round256(bc_row * rows);
    const size_t cst = last_state ? round256(st_ch * cd * rows) : 0;
    const size_t per_set = cact * (z ? 4 : 3) + 2 * cbc + cst;
    const size_t total = szA + szD + szb + per_set * nset;
    uint8_t* base = nullptr;
    if (fault_alloc() ||
        cudaMallocAsync(reinterpret_cast<void**>(&base), total, s0) != cudaSuccess) {
        cudaGetLastError();
        return SS_ERR_ALLOC;
    }
    int rc = SS_OK;
    cudaEvent_t ev_start = nullptr, ev_end = nullptr;
    auto H2D = [&](void* dst, const void* src, size_t n, cudaStream_t st) {
        if (n && rc == SS_OK && cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, st) != cudaSuccess)
            rc = SS_ERR_CUDA;
    };
    auto D2H = [&](void* dst, const void* src, size_t n, cudaStream_t st) {
        if (n && rc == SS_OK && cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, st) != cudaSuccess)
            rc = SS_ERR_CUDA;
    };
    float* dA = reinterpret_cast<float*>(base);
    float* dD = D ? reinterpret_cast<float*>(base + szA) : nullptr;
    float* dbias = delta_bias ? reinterpret_cast<float*>(base + szA + szD) : nullptr;
    H2D(dA, A->data, numel(A) * sizeof(float), s0);
    if (D) H2D(dD, D->data, Dch * sizeof(float), s0);
    if (delta_bias) H2D(dbias, delta_bias->data, Dch * sizeof(float), s0);
    if (rc == SS_OK && (cudaEventCreateWithFlags(&ev_start, cudaEventDisableTiming) != cudaSuccess ||
                        cudaEventCreateWithFlags(&ev_end, cudaEventDisableTiming) != cudaSuccess ||
                        cudaEventRecord(ev_start, s0) != cudaSuccess ||
                        cudaStreamWaitEvent(s1, ev_start, 0) != cudaSuccess))
        rc = SS_ERR_CUDA;
    Scratch sc{scratch_alloc_async, scratch_free_async, nullptr};
    int64_t set_row[2] = {-1, -1};  // batch row whose B, C a set holds (channel blocks)
    for (int64_t i = 0; i < nchunk && rc == SS_OK; ++i) {
        // rows [b0, b0 + nb) of channels [d0, d0 + nd)
        int64_t b0, nb, d0, nd;
        if (cd < Dch) {
            b0 = i / cblocks; nb = 1;
            d0 = (i % cblocks) * cd; nd = std::min(cd, Dch - d0);
        } else {
            b0 = i * rows; nb = std::min(rows, Bsz - b0);
            d0 = 0; nd = Dch;
        }
        const int si = (int)(i % nset);
        cudaStream_t st = (i % 2 == 0) ? s0 : s1;
        uint8_t* set = base + szA + szD + szb + per_set * si;
        uint8_t *du = set, *ddl = set + cact, *dy = set + 2 * cact;
        uint8_t* dz = z ? set + 3 * cact : nullptr;
        uint8_t* dB = set + cact * (z ? 4 : 3);
        uint8_t* dC = dB + cbc;
        float* dlast = last_state ? reinterpret_cast<float*>(dC + cbc) : nullptr;
        // inputs: rows (or one row's channel block) are contiguous in every tensor
        const size_t off_act = ((size_t)b0 * Dch + d0) * act_ch, n_act = (size_t)nb * nd * act_ch;
        H2D(du, static_cast<const uint8_t*>(u->data) + off_act, n_act, st);
        H2D(ddl, static_cast<const uint8_t*>(delta->data) + off_act, n_act, st);
        if (z) H2D(dz, static_cast<const uint8_t*>(z->data) + off_act, n_act, st);
        if (cd == Dch || set_row[si] != b0) {  // a channel block reuses its row's B, C
            H2D(dB, static_cast<const uint8_t*>(B->data) + (size_t)b0 * bc_row, bc_row * nb, st);
            H2D(dC, static_cast<const uint8_t*>(C->data) + (size_t)b0 * bc_row, bc_row * nb, st);
            set_row[si] = b0;
        }
        if (rc != SS_OK) break;
        ScanArgs c = a;  // contiguous rows: the strides stay, the pointers move
        c.Bsz = (int)nb;
        c.D = (int)nd;
        c.u = du; c.dl = ddl; c.z = dz; c.y = dy;
        c.A = dA + d0 * a.sA_d; c.Dv = dD ? dD + d0 * a.sD : nullptr;
        c.bias = dbias ? dbias + d0 * a.sbias : nullptr; c.last = dlast;
        if (G > 1) {  // the block's groups only
            const int64_t gsz = Dch / G;
            c.G = (int)(nd / gsz);
            c.Bm = dB + (size_t)(d0 / gsz) * a.sB_g * es;
            c.Cm = dC + (size_t)(d0 / gsz) * a.sC_g * es;
            if (nb == 1) {  // one row: its groups are evenly spaced, as the TMA map expects
                c.sB_b = c.G * a.sB_g;
                c.sC_b = c.G * a.sC_g;
            }
        } else {
            c.Bm = dB; c.Cm = dC;
        }
        rc = launch_selective(c, st, sc);
        if (rc != SS_OK) break;
        D2H(static_cast<uint8_t*>(y->data) + off_act, dy, n_act, st);
        if (last_state)
            D2H(static_cast<uint8_t*>(last_state->data) + ((size_t)b0 * Dch + d0) * st_ch, dlast,
                (size_t)nb * nd * st_ch, st);
    }
    // join the side stream back into the caller's stream, then free
    if (ev_end && (cudaEventRecord(ev_end, s1) != cudaSuccess ||
                   cudaStreamWaitEvent(s0, ev_end, 0) != cudaSuccess) && rc == SS_OK)
        rc = SS_ERR_CUDA;
    cudaFreeAsync(base, s0);
    if (ev_start) cudaEventDestroy(ev_start);
    if (ev_end) cudaEventDestroy(ev_end);
    return rc;
}

// Checks the arguments of an SSD call and fills `a` (pointers as given: the
// host-buffer entry point uses it for the shapes and strides only); *nothing
// is set when the call has no work.
static int ssd_args(const ss_tensor* x, const ss_tensor* dt, const ss_tensor* A_head,
                    const ss_tensor* B, const ss_tensor* C, const ss_tensor* D, int chunk,
                    const ss_tensor* h0, ss_tensor* y, ss_tensor* last_state, SSDArgs* out,
                    bool* nothing) {
    *nothing = false;
    SS_TRY(check_tensor(x, 4));
    SS_TRY(check_tensor(dt, 3));
    SS_TRY(check_tensor(A_head, 1));
    SS_TRY(check_tensor(B, 4));
    SS_TRY(check_tensor(C, 4));
    SS_TRY(check_tensor(y, 4));
    if (D) SS_TRY(check_tensor(D, 1));
    if (last_state) SS_TRY(check_tensor(last_state, 4));
    if (h0) SS_TRY(check_tensor(h0, 4));
    if (chunk != 64 && chunk != 128 && chunk != 256) return SS_ERR_INVALID_ARG;
    const int ty = x->dtype;
    if (dt->dtype != ty || B->dtype != ty || C->dtype != ty || y->dtype != ty) return SS_ERR_DTYPE;
    if (A_head->dtype != SS_F32 || (D && D->dtype != SS_F32) ||
        (last_state && last_state->dtype != SS_F32) || (h0 && h0->dtype != SS_F32))
        return SS_ERR_DTYPE;
    const int64_t Bsz = x->shape[0], L = x->shape[1], H = x->shape[2], P = x->shape[3];
    const int64_t G = B->shape[2], N = B->shape[3];
    if (!same_shape(y, x)) return SS_ERR_SHAPE;
    if (dt->shape[0] != Bsz || dt->shape[1] != L || dt->shape[2] != H) return SS_ERR_SHAPE;
    if (A_head->shape[0] != H || (D && D->shape[0] != H)) return SS_ERR_SHAPE;
    if (B->shape[0] != Bsz || B->shape[1] != L || !same_shape(C, B)) return SS_ERR_SHAPE;
    if (G < 1 || N < 1 || H % G != 0) return SS_ERR_SHAPE;
    if (last_state && (last_state->shape[0] != Bsz || last_state->shape[1] != H ||
                       last_state->shape[2] != P || last_state->shape[3] != N))
        return SS_ERR_SHAPE;
    if (h0 && (h0->shape[0] != Bsz || h0->shape[1] != H || h0->shape[2] != P || h0->shape[3] != N))
        return SS_ERR_SHAPE;
    if (N > 256 || P > 1024) return SS_ERR_UNSUPPORTED;
    if (Bsz * H * P >= (int64_t(1) << 31) || L >= (int64_t(1) << 31)) return SS_ERR_UNSUPPORTED;
    if (Bsz == 0 || H == 0 || P == 0 || (L == 0 && !last_state)) {
        *nothing = true;
        return SS_OK;
    }

    SSDArgs& a = *out;
    a = SSDArgs{};
    a.Bsz = (int)Bsz; a.L = (int)L; a.H = (int)H; a.P = (int)P; a.G = (int)G; a.N = (int)N;
    a.chunk = chunk; a.dtype = ty;
    a.x = x->data; a.sx_b = x->stride[0]; a.sx_l = x->stride[1]; a.sx_h = x->stride[2]; a.sx_p = x->stride[3];
    a.dt = dt->data; a.sdt_b = dt->stride[0]; a.sdt_l = dt->stride[1]; a.sdt_h = dt->stride[2];
    a.A = static_cast<const float*>(A_head->data); a.sA = A_head->stride[0];
    a.Bm = B->data; a.sB_b = B->stride[0]; a.sB_l = B->stride[1]; a.sB_g = B->stride[2]; a.sB_n = B->stride[3];
    a.Cm = C->data; a.sC_b = C->stride[0]; a.sC_l = C->stride[1]; a.sC_g = C->stride[2]; a.sC_n = C->stride[3];
    if (D) { a.Dv = static_cast<const float*>(D->data); a.sD = D->stride[0]; }
    a.y = y->data; a.sy_b = y->stride[0]; a.sy_l = y->stride[1]; a.sy_h = y->stride[2]; a.sy_p = y->stride[3];
    if (last_state) {
        a.last = static_cast<float*>(last_state->data);
        a.sl_b = last_state->stride[0]; a.sl_h = last_state->stride[1];
        a.sl_p = last_state->stride[2]; a.sl_n = last_state->stride[3];
    }
    if (h0) {
        a.h0 = static_cast<const float*>(h0->data);
        a.sh_b = h0->stride[0]; a.sh_h = h0->stride[1]; a.sh_p = h0->stride[2]; a.sh_n = h0->stride[3];
    }
    a.err = device_error_ptr();
    if (!a.err) return SS_ERR_CUDA;
    return SS_OK;
}

int ss_ssd_chunk_scan_fwd_init(const ss_tensor* x, const ss_tensor* dt, const ss_tensor* A_head,
                               const ss_tensor* B, const ss_tensor* C, const ss_tensor* D,
                               int chunk, const ss_tensor* initial_state, ss_tensor* y,
                               ss_tensor* last_state, void* stream) {
    SSDArgs a{};
    bool nothing = false;
    SS_TRY(ssd_args(x, dt, A_head, B, C, D, chunk, initial_state, y, last_state, &a, &nothing));
    if (nothing) return SS_OK;
    Scratch sc{scratch_alloc_async, scratch_free_async, nullptr};
    return launch_ssd(a, static_cast<cudaStream_t>(stream), sc);
}

int ss_ssd_chunk_scan_fwd(const ss_tensor* x, const ss_tensor* dt, const ss_tensor* A_head,
                          const ss_tensor* B, const ss_tensor* C, const ss_tensor* D, int chunk,
                          ss_tensor* y, ss_tensor* last_state, void* stream) {
    return ss_ssd_chunk_scan_fwd_init(x, dt, A_head, B, C, D, chunk, nullptr, y, last_state,
                                      stream);
}

// ---------------------------------------------------------------------------
// Host buffers in and out: ss_ssd_chunk_scan_fwd_host.  The batch is cut into
// chunks of batch rows, or of one row's heads (whole channel groups) when a
// row is large; chunks alternate between the caller's stream and the side
// stream as in ss_selective_scan_fwd_host.

int ss_ssd_chunk_scan_fwd_host(const ss_tensor* x, const ss_tensor* dt, const ss_tensor* A_head,
                               const ss_tensor* B, const ss_tensor* C, const ss_tensor* D,
                               int chunk, ss_tensor* y, ss_tensor* last_state, void* stream) {
    SSDArgs a{};
    bool nothing = false;
    SS_TRY(ssd_args(x, dt, A_head, B, C, D, chunk, nullptr, y, last_state, &a, &nothing));
    if (nothing) return SS_OK;
    for (const ss_tensor* t : {x, dt, A_head, B, C, D, static_cast<const ss_tensor*>(y),
                               static_cast<const ss_tensor*>(last_state)})
        if (t && !is_contiguous(t)) return SS_ERR_UNSUPPORTED;
    cudaStream_t s0 = static_cast<cudaStream_t>(stream);
    cudaStream_t s1 = side_stream();
    if (!s1) return SS_ERR_CUDA;

    const int es = elem_size(x->dtype);
    const int64_t Bsz = a.Bsz, L = a.L, H = a.H, P = a.P, G = a.G, N = a.N;
    const int64_t hpg = H / G;                       // heads per group
    const size_t head_bytes = (size_t)L * P * es;    // one head of one batch row of x or y
    const size_t row_bytes = head_bytes * H;
    const size_t bc_row = (size_t)L * G * N * es;    // one batch row of B or C
    // Chunks of about 32 MB of x: whole batch rows while a row is smaller (at
    // least two chunks when there are two rows), else blocks of one row's
    // heads, so that the copies overlap the scan: whole groups, or, when a
    // group alone is larger, the largest divisor of the heads per group that
    // fits (the block's heads then share one group's B, C).
    constexpr size_t kChunkBytes = size_t(32) << 20;
    int64_t rows = 1, nh = H;
    if (row_bytes <= kChunkBytes) {
        rows = std::max<int64_t>(1, (int64_t)(kChunkBytes / std::max<size_t>(row_bytes, 1)));
        if (Bsz >= 2) rows = std::min<int64_t>(rows, (Bsz + 1) / 2);
        rows = std::min<int64_t>(rows, Bsz);
    } else {
        const int64_t want = std::max<int64_t>(1, (int64_t)(kChunkBytes / std::max<size_t>(head_bytes, 1)));
        if (want >= hpg) {
            nh = std::min<int64_t>(H, want / hpg * hpg);
        } else {
            nh = 1;
            for (int64_t d = want; d > 1; --d)
                if (hpg % d == 0) {
                    nh = d;
                    break;
                }
        }
    }
    const int64_t hblocks = (H + nh - 1) / nh;       // head blocks per batch row (whole groups each)
    const int64_t nchunk = nh < H ? Bsz * hblocks : (Bsz + rows - 1) / rows;
    const int nset = nchunk > 1 ? 2 : 1;
    const int64_t dtp = (nh + 7) / 8 * 8;            // dt's t-pitch on the device: a multiple of 8

    // device layout: A_head, D once; then `nset` sets of chunk buffers
    const size_t szA = round256(H * sizeof(float)), szD = D ? round256(H * sizeof(float)) : 0;
    const size_t cx = round256((size_t)rows * L * nh * P * es);
    const size_t cdt = round256((size_t)rows * L * dtp * es);
    const size_t cbc = round256(bc_row * rows);
    const size_t cst = last_state ? round256((size_t)rows * nh * P * N * sizeof(float)) : 0;
    const size_t per_set = 2 * cx + cdt + 2 * cbc + cst;
    const size_t total = szA + szD + per_set * nset;
    uint8_t* base = nullptr;
    if (fault_alloc() ||
        cudaMallocAsync(reinterpret_cast<void**>(&base), total, s0) != cudaSuccess) {
        cudaGetLastError();
        return SS_ERR_ALLOC;
    }
    int rc = SS_OK;
    cudaEvent_t ev_start = nullptr, ev_end = nullptr;
    auto copy = [&](void* dst, const void* src, size_t n, cudaMemcpyKind kind, cudaStream_t st) {
        if (n && rc == SS_OK && cudaMemcpyAsync(dst, src, n, kind, st) != cudaSuccess) rc = SS_ERR_CUDA;
    };
    auto copy2d = [&](void* dst, size_t dpitch, const void* src, size_t spitch, size_t width,
                      size_t height, cudaMemcpyKind kind, cudaStream_t st) {
        if (width && height && rc == SS_OK &&
            cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, height, kind, st) != cudaSuccess)
            rc = SS_ERR_CUDA;
    };
    float* dA = reinterpret_cast<float*>(base);
    float* dD = D ? reinterpret_cast<float*>(base + szA) : nullptr;
    copy(dA, A_head->data, H * sizeof(float), cudaMemcpyHostToDevice, s0);
    if (D) copy(dD, D->data, H * sizeof(float), cudaMemcpyHostToDevice, s0);
    if (rc == SS_OK && (cudaEventCreateWithFlags(&ev_start, cudaEventDisableTiming) != cudaSuccess ||
                        cudaEventCreateWithFlags(&ev_end, cudaEventDisableTiming) != cudaSuccess ||
                        cudaEventRecord(ev_start, s0) != cudaSuccess ||
                        cudaStreamWaitEvent(s1, ev_start, 0) != cudaSuccess))
        rc = SS_ERR_CUDA;
    Scratch sc{scratch_alloc_async, scratch_free_async, nullptr};
    int64_t set_row[2] = {-1, -1};  // batch row whose B, C a set holds (head blocks)
    const uint8_t* xh = static_cast<const uint8_t*>(x->data);
    const uint8_t* dth = static_cast<const uint8_t*>(dt->data);
    for (int64_t i = 0; i < nchunk && rc == SS_OK; ++i) {
        // rows [b0, b0 + nb) of heads [hb, hb + nhc)
        int64_t b0, nb, hb, nhc;
        if (nh < H) {
            b0 = i / hblocks; nb = 1;
            hb = (i % hblocks) * nh; nhc = std::min(nh, H - hb);
        } else {
            b0 = i * rows; nb = std::min(rows, Bsz - b0);
            hb = 0; nhc = H;
        }
        const int si = (int)(i % nset);
        cudaStream_t st = (i % 2 == 0) ? s0 : s1;
        uint8_t* set = base + szA + szD + per_set * si;
        uint8_t *dx = set, *dy = set + cx, *ddt = set + 2 * cx;
        uint8_t* dB = ddt + cdt;
        uint8_t* dC = dB + cbc;
        float* dlast = last_state ? reinterpret_cast<float*>(dC + cbc) : nullptr;
        // x: (nb * L) rows of nhc heads, pitch H heads on the host
        const size_t hw = (size_t)nhc * P * es, hp = (size_t)H * P * es;
        const size_t off_x = ((size_t)b0 * L * H + hb) * P * es;
        if (nhc == H) copy(dx, xh + off_x, (size_t)nb * row_bytes, cudaMemcpyHostToDevice, st);
        else copy2d(dx, hw, xh + off_x, hp, hw, (size_t)nb * L, cudaMemcpyHostToDevice, st);
        // dt: (nb * L) rows of nhc values, to a pitch of dtp values
        copy2d(ddt, (size_t)dtp * es, dth + ((size_t)b0 * L * H + hb) * es, (size_t)H * es,
               (size_t)nhc * es, (size_t)nb * L, cudaMemcpyHostToDevice, st);
        if (nh == H || set_row[si] != b0) {  // a head block reuses its row's B, C
            copy(dB, static_cast<const uint8_t*>(B->data) + (size_t)b0 * bc_row, bc_row * nb,
                 cudaMemcpyHostToDevice, st);
            copy(dC, static_cast<const uint8_t*>(C->data) + (size_t)b0 * bc_row, bc_row * nb,
                 cudaMemcpyHostToDevice, st);
            set_row[si] = b0;
        }
        if (rc != SS_OK) break;
        SSDArgs c = a;  // the chunk's tensors are contiguous (dt padded)
        c.Bsz = (int)nb;
        c.H = (int)nhc;
        c.G = (int)(nhc >= hpg ? nhc / hpg : 1);  // whole groups, or part of one
        c.x = dx; c.sx_b = L * nhc * P; c.sx_l = nhc * P; c.sx_h = P; c.sx_p = 1;
        c.y = dy; c.sy_b = L * nhc * P; c.sy_l = nhc * P; c.sy_h = P; c.sy_p = 1;
        c.dt = ddt; c.sdt_b = L * dtp; c.sdt_l = dtp; c.sdt_h = 1;
        const int64_t g0 = hb / hpg;  // the block's first group
        c.Bm = dB + (size_t)g0 * N * es; c.sB_b = L * G * N; c.sB_l = G * N; c.sB_g = N; c.sB_n = 1;
        c.Cm = dC + (size_t)g0 * N * es; c.sC_b = L * G * N; c.sC_l = G * N; c.sC_g = N; c.sC_n = 1;
        c.A = dA + hb; c.sA = 1;
        c.Dv = dD ? dD + hb : nullptr; c.sD = 1;
        c.last = dlast; c.sl_b = nhc * P * N; c.sl_h = P * N; c.sl_p = N; c.sl_n = 1;
        c.h0 = nullptr;
        rc = launch_ssd(c, st, sc);
        if (rc != SS_OK) break;
        uint8_t* yh = static_cast<uint8_t*>(y->data);
        if (nhc == H) copy(yh + off_x, dy, (size_t)nb * row_bytes, cudaMemcpyDeviceToHost, st);
        else copy2d(yh + off_x, hp, dy, hw, hw, (size_t)nb * L, cudaMemcpyDeviceToHost, st);
        if (last_state)
            copy(static_cast<uint8_t*>(last_state->data) + ((size_t)b0 * H + hb) * P * N * sizeof(float),
                 dlast, (size_t)nb * nhc * P * N * sizeof(float), cudaMemcpyDeviceToHost, st);
    }
    // join the side stream back into the caller's stream, then free
    if (ev_end && (cudaEventRecord(ev_end, s1) != cudaSuccess ||
                   cudaStreamWaitEvent(s0, ev_end, 0) != cudaSuccess) && rc == SS_OK)
        rc = SS_ERR_CUDA;
    cudaFreeAsync(base, s0);
    if (ev_start) cudaEventDestroy(ev_start);
    if (ev_end) cudaEventDestroy(ev_end);
    return rc;
}

int ss_selective_state_update(ss_tensor* state, const ss_tensor* u, const ss_tensor* delta,
                              const ss_tensor* A, const ss_tensor* B, const ss_tensor* C,
                              const ss_tensor* D, const ss_tensor* z, const ss_tensor* delta_bias,
                              int softplus, ss_tensor* y, void* stream) {
    SS_TRY(check_tensor(state, 3));
    SS_TRY(check_tensor(u, 2));
    SS_TRY(check_tensor(delta, 2));
    SS_TRY(check_tensor(A, 2));
    SS_TRY(check_tensor(B, 2));
    SS_TRY(check_tensor(C, 2));
    SS_TRY(check_tensor(y, 2));
    if (D) SS_TRY(check_tensor(D, 1));
    if (z) SS_TRY(check_tensor(z, 2));
    if (delta_bias) SS_TRY(check_tensor(delta_bias, 1));
    if (softplus != 0 && softplus != 1) return SS_ERR_INVALID_ARG;
    const int ty = u->dtype;
    if (delta->dtype != ty || B->dtype != ty || C->dtype != ty || y->dtype != ty ||
        (z && z->dtype != ty))
        return SS_ERR_DTYPE;
    if (state->dtype != SS_F32 || A->dtype != SS_F32 || (D && D->dtype != SS_F32) ||
        (delta_bias && delta_bias->dtype != SS_F32))
        return SS_ERR_DTYPE;
    const int64_t Bsz = u->shape[0], Dch = u->shape[1], N = A->shape[1];
    if (!same_shape(delta, u) || !same_shape(y, u) || (z && !same_shape(z, u))) return SS_ERR_SHAPE;
    if (A->shape[0] != Dch || B->shape[0] != Bsz || B->shape[1] != N || !same_shape(C, B))
        return SS_ERR_SHAPE;
    if (state->shape[0] != Bsz || state->shape[1] != Dch || state->shape[2] != N) return SS_ERR_SHAPE;
    if ((D && D->shape[0] != Dch) || (delta_bias && delta_bias->shape[0] != Dch)) return SS_ERR_SHAPE;
    if (N < 1) return SS_ERR_SHAPE;
    if (N > 256) return SS_ERR_UNSUPPORTED;
    if (Bsz * Dch >= (int64_t(1) << 31)) return SS_ERR_UNSUPPORTED;
    if (Bsz == 0 || Dch == 0) return SS_OK;
    StepArgs a{};
    a.Bsz = (int)Bsz; a.D = (int)Dch; a.N = (int)N; a.dtype = ty;
    a.state = static_cast<float*>(state->data);
    a.ss_b = state->stride[0]; a.ss_d = state->stride[1]; a.ss_n = state->stride[2];
    a.u = u->data; a.su_b = u->stride[0]; a.su_d = u->stride[1];
    a.dl = delta->data; a.sdl_b = delta->stride[0]; a.sdl_d = delta->stride[1];
    if (z) { a.z = z->data; a.sz_b = z->stride[0]; a.sz_d = z->stride[1]; }
    a.y = y->data; a.sy_b = y->stride[0]; a.sy_d = y->stride[1];
    a.Bm = B->data; a.sB_b = B->stride[0]; a.sB_n = B->stride[1];
    a.Cm = C->data; a.sC_b = C->stride[0]; a.sC_n = C->stride[1];
    a.A = static_cast<const float*>(A->data); a.sA_d = A->stride[0]; a.sA_n = A->stride[1];
    if (D) { a.Dv = static_cast<const float*>(D->data); a.sD = D->stride[0]; }
    if (delta_bias) { a.bias = static_cast<const float*>(delta_bias->data); a.sbias = delta_bias->stride[0]; }
    a.softplus = softplus;
    return launch_selective_step(a, static_cast<cudaStream_t>(stream));
}

int ss_ssd_state_update(ss_tensor* state, const ss_tensor* x, const ss_tensor* dt,
                        const ss_tensor* A_head, const ss_tensor* B, const ss_tensor* C,
                        const ss_tensor* D, ss_tensor* y, void* stream) {
    SS_TRY(check_tensor(state, 4));
    SS_TRY(check_tensor(x, 3));
    SS_TRY(check_tensor(dt, 2));
    SS_TRY(check_tensor(A_head, 1));
    SS_TRY(check_tensor(B, 3));
    SS_TRY(check_tensor(C, 3));
    SS_TRY(check_tensor(y, 3));
    if (D) SS_TRY(check_tensor(D, 1));
    const int ty = x->dtype;
    if (dt->dtype != ty || B->dtype != ty || C->dtype != ty || y->dtype != ty) return SS_ERR_DTYPE;
    if (state->dtype != SS_F32 || A_head->dtype != SS_F32 || (D && D->dtype != SS_F32))
        return SS_ERR_DTYPE;
    const int64_t Bsz = x->shape[0], H = x->shape[1], P = x->shape[2];
    const int64_t G = B->shape[1], N = B->shape[2];
    if (!same_shape(y, x) || dt->shape[0] != Bsz || dt->shape[1] != H) return SS_ERR_SHAPE;
    if (A_head->shape[0] != H || (D && D->shape[0] != H)) return SS_ERR_SHAPE;
    if (B->shape[0] != Bsz || !same_shape(C, B) || G < 1 || N < 1 || H % G != 0) return SS_ERR_SHAPE;
    if (state->shape[0] != Bsz || state->shape[1] != H || state->shape[2] != P ||
        state->shape[3] != N)
        return SS_ERR_SHAPE;
    if (N > 256 || P > 1024) return SS_ERR_UNSUPPORTED;
    if (Bsz * H * P >= (int64_t(1) << 26)) return SS_ERR_UNSUPPORTED;
    if (Bsz == 0 || H == 0 || P == 0) return SS_OK;
    SSDStepArgs a{};
    a.Bsz = (int)Bsz; a.H = (int)H; a.P = (int)P; a.G = (int)G; a.N = (int)N; a.dtype = ty;
    a.state = static_cast<float*>(state->data);
    a.ss_b = state->stride[0]; a.ss_h = state->stride[1]; a.ss_p = state->stride[2]; a.ss_n = state->stride[3];
    a.x = x->data; a.sx_b = x->stride[0]; a.sx_h = x->stride[1]; a.sx_p = x->stride[2];
    a.dt = dt->data; a.sdt_b = dt->stride[0]; a.sdt_h = dt->stride[1];
    a.A = static_cast<const float*>(A_head->data); a.sA = A_head->stride[0];
    a.Bm = B->data; a.sB_b = B->stride[0]; a.sB_g = B->stride[1]; a.sB_n = B->stride[2];
    a.Cm = C->data; a.sC_b = C->stride[0]; a.sC_g = C->stride[1]; a.sC_n = C->stride[2];
    if (D) { a.Dv = static_cast<const float*>(D->data); a.sD = D->stride[0]; }
    a.y = y->data; a.sy_b = y->stride[0]; a.sy_h = y->stride[1]; a.sy_p = y->stride[2];
    return launch_ssd_step(a, static_cast<cudaStream_t>(stream));
}

const char* ss_status_string(int status) {
    switch (status) {
        case SS_OK: return "ok";
        case SS_ERR_INVALID_ARG: return "invalid argument";
        case SS_ERR_SHAPE: return "shape mismatch";
        case SS_ERR_DTYPE: return "unsupported or mixed dtype";
        case SS_ERR_ALIGNMENT: return "misaligned pointer";
        case SS_ERR_UNSUPPORTED: return "unsupported size";
        case SS_ERR_ALLOC: return "scratch allocation failed";
        case SS_ERR_LAUNCH: return "kernel launch failed";
        case SS_ERR_TIMEOUT: return "device-side wait timed out";
        case SS_ERR_CUDA: return "CUDA runtime error";
        default: return "unknown status";
    }
}

int ss_get_device_error(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SS_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return SS_ERR_CUDA;
    if (v) {
        const unsigned zero = 0;
        cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
        return SS_ERR_TIMEOUT;
    }
    return SS_OK;
}

int ss_selftest_timeout(unsigned limit_us, void* stream) {
    if (limit_us < 1 || limit_us > 100000) return SS_ERR_INVALID_ARG;
    unsigned* err = device_error_ptr();
    if (!err) return SS_ERR_CUDA;
    return launch_selftest_wait(limit_us, err, static_cast<cudaStream_t>(stream));
}

int ss_probe_ex2_rate(double* ex2_per_sm_per_clock, void* stream) {
    if (!ex2_per_sm_per_clock) return SS_ERR_INVALID_ARG;
    return probe_ex2_rate(ex2_per_sm_per_clock, static_cast<cudaStream_t>(stream));
}

int ss_probe_scan_forms(double* seq_steps_per_s, double* shfl_steps_per_s, void* stream) {
    if (!seq_steps_per_s || !shfl_steps_per_s) return SS_ERR_INVALID_ARG;
    return probe_scan_forms(seq_steps_per_s, shfl_steps_per_s, static_cast<cudaStream_t>(stream));
}

uint64_t ss_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int ss_version(void) { return 300; }

}  // extern "C"
