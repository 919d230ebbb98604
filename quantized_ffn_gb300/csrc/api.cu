// api.cu -- the C ABI: host-side argument checks, per-device state (error
// word, workspace), and the choice between the single-token kernel and the
// tensor-core kernel.  Every step of the computation runs in this library's
// kernels; there is no host fallback.
#include <mutex>

#include "zffn_internal.cuh"
#include "formats.h"
#include "rmsnorm.h"
#include "router.h"

namespace zffn {

static __device__ int g_device_error;   // one per device that loads the library

namespace {

constexpr int kMaxDevices = 64;

struct Workspace {
    void *ptr = nullptr;
    size_t bytes = 0;
};

std::mutex g_mu;
DeviceInfo g_info[kMaxDevices];
Workspace g_ws[kMaxDevices];
int g_matvec_max_t = 1;
int g_moe_kernel = 0;   // ZFFN_OPT_MOE_KERNEL
int g_token_kernel = 0; // ZFFN_OPT_TOKEN_KERNEL

thread_local const char *t_last_error = "no error";   // zffn_last_error()

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Sub-buffers carved out of one device allocation.
struct Layout {
    size_t gbar, h, counts, offsets, cursors, tiles, n_tiles, row_token, row_weight, x_perm, xn, x16,
        total;
    int max_tiles;
};

Layout layout_for(int T, int H, int I, int E, int k) {
    Layout L;
    size_t o = 0;
    const int64_t P = (int64_t)T * k;
    // tiles of at least 32 rows (the grouped kernel's groups; 128 otherwise)
    L.max_tiles = (int)((P + 31) / 32 + (E < P ? E : P));
    // the grid barrier of the one-launch routed path: first, so that it keeps
    // its place (and its zero state) whatever the sizes of a call
    L.gbar = o; o = align_up(o + sizeof(unsigned long long));
    L.h = o; o = align_up(o + (size_t)P * I * sizeof(float));
    L.counts = o; o = align_up(o + (size_t)E * sizeof(int));
    L.offsets = o; o = align_up(o + (size_t)(E + 1) * sizeof(int));
    L.cursors = o; o = align_up(o + (size_t)E * sizeof(int));
    L.tiles = o; o = align_up(o + (size_t)L.max_tiles * sizeof(int4));
    L.n_tiles = o; o = align_up(o + sizeof(int));
    L.row_token = o; o = align_up(o + (size_t)P * sizeof(int));
    L.row_weight = o; o = align_up(o + (size_t)P * sizeof(float));
    L.x_perm = o; o = align_up(o + (size_t)P * H * 2);
    L.xn = o; o = align_up(o + (size_t)T * H * 2);      // normalised block input (pre-norm entry)
    L.x16 = o; o = align_up(o + (size_t)T * H * 2);     // fp16 block input of the tensor-core path
    L.total = o;
    return L;
}

int current_device() {
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess) return -1;
    return d;
}

// Make sure the current device's workspace holds at least `bytes`.
zffn_status ensure_workspace(size_t bytes, Workspace **out) {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) {
        t_last_error = "no usable CUDA device";
        return ZFFN_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    Workspace &w = g_ws[dev];
    if (w.bytes < bytes) {
        if (w.ptr) {
            // the old buffer may still be in use by queued work on the device
            if (cudaDeviceSynchronize() != cudaSuccess) return ZFFN_ERR_CUDA;
            cudaFree(w.ptr);
            w = Workspace{};
        }
        void *p = nullptr;
        if (cudaMalloc(&p, bytes) != cudaSuccess) {
            cudaGetLastError();
            return ZFFN_ERR_NO_WORKSPACE;
        }
        // the barrier words (and everything else) start at zero, before any
        // stream can use the buffer
        if (cudaMemset(p, 0, bytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
            cudaFree(p);
            cudaGetLastError();
            return ZFFN_ERR_CUDA;
        }
        w.ptr = p;
        w.bytes = bytes;
    }
    *out = &w;
    return ZFFN_OK;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// A failed host-side check: record why (zffn_last_error) and return INVALID_ARG.
zffn_status invalid(const char *why) {
    t_last_error = why;
    return ZFFN_ERR_INVALID_ARG;
}

zffn_status check_shape(int T, int H, int I) {
    if (T < 1) return invalid("T must be at least 1");
    if (H < 256 || H > 16384 || H % 256 != 0)
        return invalid("H must be a multiple of 256 in [256, 16384]");
    if (I < 64 || I > 65536 || I % 64 != 0) return invalid("I must be a multiple of 64 in [64, 65536]");
    return ZFFN_OK;
}

zffn_status to_status(cudaError_t e) {
    if (e == cudaSuccess) return ZFFN_OK;
    t_last_error = cudaGetErrorString(e);
    cudaGetLastError();
    return ZFFN_ERR_CUDA;
}

}  // namespace

void set_last_error(const char *what) { t_last_error = what; }

namespace {
struct SmemAttr {
    const void *fn;
    int device;
    size_t bytes;
};
std::mutex g_attr_mu;
SmemAttr g_attr[256];
int g_attr_n = 0;
}  // namespace

cudaError_t ensure_dynamic_smem(const void *fn, size_t bytes) {
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    SmemAttr *rec = nullptr;
    for (int i = 0; i < g_attr_n; ++i)
        if (g_attr[i].fn == fn && g_attr[i].device == dev) rec = &g_attr[i];
    if (rec && rec->bytes >= bytes) return cudaSuccess;
    if (!rec && g_attr_n == (int)(sizeof(g_attr) / sizeof(g_attr[0]))) return cudaErrorMemoryAllocation;
    const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    if (!rec) {
        rec = &g_attr[g_attr_n++];
        rec->fn = fn;
        rec->device = dev;
    }
    rec->bytes = bytes;
    return cudaSuccess;
}

namespace {
// No usable device: record why for zffn_last_error and hand back the empty
// record (device -1), which every entry turns into ZFFN_ERR_CUDA.
const DeviceInfo &no_device(cudaError_t e) {
    static const DeviceInfo none;
    t_last_error = e == cudaSuccess ? "device index beyond the library's device table"
                                    : cudaGetErrorString(e);
    cudaGetLastError();
    return none;
}
}  // namespace

const DeviceInfo &device_info() {
    int dev = -1;
    const cudaError_t ge = cudaGetDevice(&dev);
    if (ge != cudaSuccess || dev < 0 || dev >= kMaxDevices) return no_device(ge);
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &di = g_info[dev];
    if (di.device != dev) {
        cudaDeviceProp prop;
        cudaError_t e = cudaGetDeviceProperties(&prop, dev);
        if (e != cudaSuccess) return no_device(e);
        di.num_sms = prop.multiProcessorCount;
        di.max_smem_optin = (int)prop.sharedMemPerBlockOptin;
        void *addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_device_error);
        if (e != cudaSuccess) return no_device(e);
        di.err_word = static_cast<int *>(addr);
        di.device = dev;
    }
    return di;
}

}  // namespace zffn

using namespace zffn;

extern "C" {

const char *zffn_status_string(zffn_status s) {
    switch (s) {
        case ZFFN_OK: return "ZFFN_OK";
        case ZFFN_ERR_INVALID_ARG: return "ZFFN_ERR_INVALID_ARG";
        case ZFFN_ERR_UNSUPPORTED: return "ZFFN_ERR_UNSUPPORTED";
        case ZFFN_ERR_CUDA: return "ZFFN_ERR_CUDA";
        case ZFFN_ERR_TIMEOUT: return "ZFFN_ERR_TIMEOUT";
        case ZFFN_ERR_NO_WORKSPACE: return "ZFFN_ERR_NO_WORKSPACE";
    }
    return "ZFFN_UNKNOWN_STATUS";
}

size_t zffn_q4k_row_bytes(int64_t cols) {
    return cols <= 0 ? 0 : (size_t)q4k_row_bytes(cols);
}

zffn_status zffn_q4k_dequant(const void *blocks, float *out, int64_t rows, int64_t cols,
                             void *stream) {
    if (!blocks || !out) return invalid("a pointer argument is NULL");
    if (rows <= 0 || cols <= 0) return invalid("rows and cols must be positive");
    if (device_info().device < 0) return ZFFN_ERR_CUDA;
    return to_status(launch_q4k_dequant(blocks, out, rows, cols, (cudaStream_t)stream));
}

zffn_status zffn_q4k_quantize(const float *w, void *blocks, int64_t rows, int64_t cols,
                              void *stream) {
    if (!w || !blocks) return invalid("a pointer argument is NULL");
    if (rows <= 0 || cols <= 0) return invalid("rows and cols must be positive");
    if (device_info().device < 0) return ZFFN_ERR_CUDA;
    return to_status(launch_q4k_quantize(w, blocks, rows, cols, (cudaStream_t)stream));
}

}  // extern "C"

namespace {

zffn_status swiglu_dense(const void *x, const void *Wg, const void *Wu, const void *Wd, float *y,
                         int T, int H, int I, void *stream, bool accumulate) {
    if (!x || !Wg || !Wu || !Wd || !y) return invalid("a pointer argument is NULL");
    if (check_shape(T, H, I) != ZFFN_OK) return ZFFN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(Wd) || !aligned16(y))
        return invalid("x, Wg, Wu, Wd and y must be 16-byte aligned");
    const DeviceInfo &di = device_info();
    if (di.device < 0) return ZFFN_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    int mv_max;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        mv_max = g_matvec_max_t;
    }
    if (T == 1 && mv_max >= 1 && matvec_smem_bytes(T, H, I, 1) <= (size_t)di.max_smem_optin) {
        const Layout L = layout_for(T, H, I, 1, 1);
        Workspace *w = nullptr;
        zffn_status st = ensure_workspace(L.total, &w);
        if (st != ZFFN_OK) return st;
        uint8_t *base = static_cast<uint8_t *>(w->ptr);
        MatvecArgs a{};
        a.x = static_cast<const __nv_bfloat16 *>(x);
        a.Wg = static_cast<const uint8_t *>(Wg);
        a.Wu = static_cast<const uint8_t *>(Wu);
        a.Wd = static_cast<const uint8_t *>(Wd);
        a.ids = nullptr;
        a.wts = nullptr;
        a.y = y;
        a.h = reinterpret_cast<float *>(base + L.h);
        a.err = di.err_word;
        a.T = T; a.H = H; a.I = I; a.E = 1; a.k = 1;
        a.accumulate = accumulate;
        return to_status(launch_ffn_matvec(a, s));
    }
    // the tensor-core kernel's gate/up operand is fp16: convert x into
    // workspace (and zero y for the kernel's reductions) in one pass
    const Layout L = layout_for(T, H, I, 1, 1);
    Workspace *w = nullptr;
    zffn_status st = ensure_workspace(L.total, &w);
    if (st != ZFFN_OK) return st;
    void *x16 = static_cast<uint8_t *>(w->ptr) + L.x16;
    cudaError_t e = launch_x_to_f16(x, x16, (int64_t)T * H, accumulate ? nullptr : y, (int64_t)T * H, s);
    if (e != cudaSuccess) return to_status(e);
    TcArgs a{};
    a.x = x16;
    a.x_rows = T;
    a.Wg = static_cast<const uint8_t *>(Wg);
    a.Wu = static_cast<const uint8_t *>(Wu);
    a.Wd = static_cast<const uint8_t *>(Wd);
    a.y = y;
    a.tiles = nullptr;
    a.n_tiles_dev = nullptr;
    a.row_token = nullptr;
    a.row_weight = nullptr;
    a.n_tiles_host = (T + 127) / 128;
    a.err = di.err_word;
    a.T = T; a.H = H; a.I = I; a.E = 1;
    return to_status(launch_ffn_tc(a, s));
}

zffn_status swiglu_moe(const void *x, const int32_t *expert_ids, const float *expert_weights,
                       const float *down_scale, const void *Wg, const void *Wu, const void *Wd,
                       float *y, int T, int H, int I, int E, int top_k, void *stream,
                       bool accumulate, int wd_fmt = kFmtQ4_K) {
    if (!x || !expert_ids || !expert_weights || !Wg || !Wu || !Wd || !y)
        return invalid("a pointer argument is NULL");
    if (check_shape(T, H, I) != ZFFN_OK) return ZFFN_ERR_INVALID_ARG;
    if (E < 1 || E > 4096 || top_k < 1 || top_k > 64)
        return invalid("E must be in [1, 4096] and top_k in [1, 64]");
    if ((int64_t)T * top_k > (1 << 24)) return invalid("T * top_k must not exceed 2^24");
    if (!aligned16(x) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(Wd) || !aligned16(y) ||
        (reinterpret_cast<uintptr_t>(expert_ids) & 3) ||
        (reinterpret_cast<uintptr_t>(expert_weights) & 3))
        return invalid("x, Wg, Wu, Wd, y must be 16-byte and expert_ids, expert_weights 4-byte aligned");
    if (reinterpret_cast<uintptr_t>(down_scale) & 3) return invalid("down_scale must be 4-byte aligned");
    const DeviceInfo &di = device_info();
    if (di.device < 0) return ZFFN_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    int mv_max, token_kernel;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        mv_max = g_matvec_max_t;
        token_kernel = g_token_kernel;
    }
    const Layout L = layout_for(T, H, I, E, top_k);
    Workspace *w = nullptr;
    zffn_status st = ensure_workspace(L.total, &w);
    if (st != ZFFN_OK) return st;
    uint8_t *base = static_cast<uint8_t *>(w->ptr);
    if (T == 1 && wd_fmt == kFmtQ4_K && mv_max >= 1 &&
        matvec_smem_bytes(T, H, I, top_k) <= (size_t)di.max_smem_optin) {
        MatvecArgs a{};
        a.x = static_cast<const __nv_bfloat16 *>(x);
        a.Wg = static_cast<const uint8_t *>(Wg);
        a.Wu = static_cast<const uint8_t *>(Wu);
        a.Wd = static_cast<const uint8_t *>(Wd);
        a.ids = expert_ids;
        a.wts = expert_weights;
        a.down_scale = down_scale;
        a.y = y;
        a.h = reinterpret_cast<float *>(base + L.h);
        a.err = di.err_word;
        a.T = T; a.H = H; a.I = I; a.E = E; a.k = top_k;
        a.accumulate = accumulate;
        a.gbar = token_kernel == 0 ? reinterpret_cast<unsigned long long *>(base + L.gbar) : nullptr;
        return to_status(launch_ffn_matvec(a, s));
    }
    // Few rows per expert: the grouped kernel (weights as the MMA's M side,
    // each Q4_K byte read once per group of 32 rows).  Many rows per expert:
    // the prefill kernel on 128-row tiles.
    int moe_kernel;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        moe_kernel = g_moe_kernel;
    }
    // (other W_down formats run on the grouped kernel only)
    const bool grouped = wd_fmt != kFmtQ4_K || moe_kernel == 1 ||
                         (moe_kernel == 0 && (int64_t)T * top_k <= (int64_t)48 * E);
    RouteArgs r{};
    r.tile_rows = grouped ? moe_group_rows() : 128;
    r.ids = expert_ids;
    r.wts = expert_weights;
    r.down_scale = down_scale;
    r.x = static_cast<const __nv_bfloat16 *>(x);
    r.T = T; r.H = H; r.E = E; r.k = top_k;
    r.counts = reinterpret_cast<int *>(base + L.counts);
    r.offsets = reinterpret_cast<int *>(base + L.offsets);
    r.cursors = reinterpret_cast<int *>(base + L.cursors);
    r.tiles = reinterpret_cast<int4 *>(base + L.tiles);
    r.n_tiles = reinterpret_cast<int *>(base + L.n_tiles);
    r.row_token = reinterpret_cast<int *>(base + L.row_token);
    r.row_weight = reinterpret_cast<float *>(base + L.row_weight);
    r.x_perm = reinterpret_cast<__half *>(base + L.x_perm);
    r.max_tiles = L.max_tiles;
    // overwrite: the gather kernel zeroes y (y is 16-byte aligned here)
    r.y_zero = accumulate ? nullptr : y;
    r.ny = (int64_t)T * H;
    cudaError_t e = launch_moe_route(r, s);
    if (e != cudaSuccess) return to_status(e);
    TcArgs a{};
    a.x = r.x_perm;
    a.x_rows = (int64_t)T * top_k;
    a.Wg = static_cast<const uint8_t *>(Wg);
    a.Wu = static_cast<const uint8_t *>(Wu);
    a.Wd = static_cast<const uint8_t *>(Wd);
    a.y = y;
    a.tiles = r.tiles;
    a.n_tiles_dev = r.n_tiles;
    a.row_token = r.row_token;
    a.row_weight = r.row_weight;
    a.n_tiles_host = L.max_tiles;
    a.err = di.err_word;
    a.T = T; a.H = H; a.I = I; a.E = E;
    return to_status(grouped ? launch_moe_group(a, wd_fmt, s) : launch_ffn_tc(a, s));
}

// The dense block with W_down in another format at T > 1: one expert on the
// grouped kernel, groups of 32 consecutive tokens (the weights are unpacked
// once per group).
zffn_status swiglu_dense_grouped(const void *x, const void *Wg, const void *Wu, const void *Wd, int wd_fmt,
                                 float *y, int T, int H, int I, void *stream, bool accumulate) {
    const DeviceInfo &di = device_info();
    if (di.device < 0) return ZFFN_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    const Layout L = layout_for(T, H, I, 1, 1);
    Workspace *w = nullptr;
    zffn_status st = ensure_workspace(L.total, &w);
    if (st != ZFFN_OK) return st;
    uint8_t *base = static_cast<uint8_t *>(w->ptr);
    int4 *tiles = reinterpret_cast<int4 *>(base + L.tiles);
    int *n_tiles = reinterpret_cast<int *>(base + L.n_tiles);
    int *row_token = reinterpret_cast<int *>(base + L.row_token);
    float *row_weight = reinterpret_cast<float *>(base + L.row_weight);
    void *x16 = base + L.x16;
    cudaError_t e = launch_dense_groups(T, moe_group_rows(), tiles, n_tiles, row_token, row_weight, s);
    if (e == cudaSuccess)
        e = launch_x_to_f16(x, x16, (int64_t)T * H, accumulate ? nullptr : y, (int64_t)T * H, s);
    if (e != cudaSuccess) return to_status(e);
    TcArgs a{};
    a.x = x16;
    a.x_rows = T;
    a.Wg = static_cast<const uint8_t *>(Wg);
    a.Wu = static_cast<const uint8_t *>(Wu);
    a.Wd = static_cast<const uint8_t *>(Wd);
    a.y = y;
    a.tiles = tiles;
    a.n_tiles_dev = n_tiles;
    a.row_token = row_token;
    a.row_weight = row_weight;
    a.n_tiles_host = (T + moe_group_rows() - 1) / moe_group_rows();
    a.err = di.err_word;
    a.T = T; a.H = H; a.I = I; a.E = 1;
    return to_status(launch_moe_group(a, wd_fmt, s));
}

}  // namespace

extern "C" {

zffn_status zffn_swiglu_q4k(const void *x, const void *Wg, const void *Wu, const void *Wd,
                            float *y, int T, int H, int I, void *stream) {
    return swiglu_dense(x, Wg, Wu, Wd, y, T, H, I, stream, false);
}

zffn_status zffn_swiglu_q4k_residual(const void *x, const void *Wg, const void *Wu,
                                     const void *Wd, float *y, int T, int H, int I,
                                     void *stream) {
    return swiglu_dense(x, Wg, Wu, Wd, y, T, H, I, stream, true);
}

zffn_status zffn_moe_swiglu_q4k(const void *x, const int32_t *expert_ids,
                                const float *expert_weights, const void *Wg, const void *Wu,
                                const void *Wd, float *y, int T, int H, int I, int E, int top_k,
                                void *stream) {
    return swiglu_moe(x, expert_ids, expert_weights, nullptr, Wg, Wu, Wd, y, T, H, I, E, top_k,
                      stream, false);
}

zffn_status zffn_moe_swiglu_q4k_residual(const void *x, const int32_t *expert_ids,
                                         const float *expert_weights, const void *Wg,
                                         const void *Wu, const void *Wd, float *y, int T, int H,
                                         int I, int E, int top_k, void *stream) {
    return swiglu_moe(x, expert_ids, expert_weights, nullptr, Wg, Wu, Wd, y, T, H, I, E, top_k,
                      stream, true);
}

size_t zffn_row_bytes_fmt(int fmt, int64_t cols) {
    return cols <= 0 || !fmt_valid(fmt) ? 0 : (size_t)fmt_row_bytes(fmt, cols);
}

zffn_status zffn_dequant_fmt(int fmt, const void *blocks, float *out, int64_t rows, int64_t cols,
                             void *stream) {
    if (!fmt_valid(fmt)) return invalid("unknown block format");
    if (!blocks || !out) return invalid("a pointer argument is NULL");
    if (rows <= 0 || cols <= 0) return invalid("rows and cols must be positive");
    if (device_info().device < 0) return ZFFN_ERR_CUDA;
    return to_status(launch_dequant_fmt(fmt, blocks, out, rows, cols, (cudaStream_t)stream));
}

}  // extern "C"

namespace {

// Routed (expert_ids != NULL) or dense block with W_down in any format, an
// optional per-expert scale of the down projection, overwrite or accumulate.
zffn_status swiglu_wd(const void *x, const int32_t *expert_ids, const float *expert_weights,
                      const float *down_scale, const void *Wg, const void *Wu, const void *Wd,
                      int wd_fmt, float *y, int T, int H, int I, int E, int top_k, void *stream,
                      bool accumulate) {
    if (!fmt_valid(wd_fmt)) return invalid("unknown block format of W_down");
    if (wd_fmt == kFmtQ4_K)
        return expert_ids ? swiglu_moe(x, expert_ids, expert_weights, down_scale, Wg, Wu, Wd, y, T,
                                       H, I, E, top_k, stream, accumulate)
                          : swiglu_dense(x, Wg, Wu, Wd, y, T, H, I, stream, accumulate);
    const bool moe = expert_ids != nullptr;
    if (!x || !Wg || !Wu || !Wd || !y || (moe && !expert_weights))
        return invalid("a pointer argument is NULL");
    if (check_shape(T, H, I) != ZFFN_OK) return ZFFN_ERR_INVALID_ARG;
    if (moe && (E < 1 || E > 4096 || top_k < 1 || top_k > 64))
        return invalid("E must be in [1, 4096] and top_k in [1, 64]");
    if (!aligned16(x) || !aligned16(Wg) || !aligned16(Wu) || (reinterpret_cast<uintptr_t>(Wd) & 3) ||
        (reinterpret_cast<uintptr_t>(y) & 3) ||
        (moe && ((reinterpret_cast<uintptr_t>(expert_ids) & 3) ||
                 (reinterpret_cast<uintptr_t>(expert_weights) & 3))))
        return invalid("x, Wg, Wu must be 16-byte and Wd, y, expert_ids, expert_weights 4-byte aligned");
    if (reinterpret_cast<uintptr_t>(down_scale) & 3) return invalid("down_scale must be 4-byte aligned");
    if (T != 1) {
        // the grouped tensor-core kernel (Q6_K rows, 210-byte blocks, are
        // bulk-copied row by row instead of through a tensor map)
        if (!aligned16(Wd) || !aligned16(y)) return invalid("for T > 1, Wd and y must be 16-byte aligned");
        if (moe)
            return swiglu_moe(x, expert_ids, expert_weights, down_scale, Wg, Wu, Wd, y, T, H, I, E, top_k,
                              stream, accumulate, wd_fmt);
        return swiglu_dense_grouped(x, Wg, Wu, Wd, wd_fmt, y, T, H, I, stream, accumulate);
    }
    const int k = moe ? top_k : 1;
    const DeviceInfo &di = device_info();
    if (di.device < 0) return ZFFN_ERR_CUDA;
    if (gu_smem_total(H, I, k) > (size_t)di.max_smem_optin ||
        down_fmt_smem_bytes(wd_fmt, I, k) > (size_t)di.max_smem_optin)
        return ZFFN_ERR_UNSUPPORTED;
    const Layout L = layout_for(1, H, I, moe ? E : 1, k);
    Workspace *w = nullptr;
    zffn_status st = ensure_workspace(L.total, &w);
    if (st != ZFFN_OK) return st;
    MatvecArgs a{};
    a.x = static_cast<const __nv_bfloat16 *>(x);
    a.Wg = static_cast<const uint8_t *>(Wg);
    a.Wu = static_cast<const uint8_t *>(Wu);
    a.Wd = static_cast<const uint8_t *>(Wd);
    a.ids = expert_ids;
    a.wts = expert_weights;
    a.down_scale = moe ? down_scale : nullptr;
    a.y = y;
    a.h = reinterpret_cast<float *>(static_cast<uint8_t *>(w->ptr) + L.h);
    a.err = di.err_word;
    a.T = 1; a.H = H; a.I = I; a.E = moe ? E : 1; a.k = k;
    a.accumulate = accumulate;
    return to_status(launch_token_fmt(a, wd_fmt, (cudaStream_t)stream));
}

}  // namespace

extern "C" {

zffn_status zffn_moe_swiglu_q4k_wd(const void *x, const int32_t *expert_ids,
                                   const float *expert_weights, const void *Wg, const void *Wu,
                                   const void *Wd, int wd_fmt, float *y, int T, int H, int I, int E,
                                   int top_k, void *stream) {
    return swiglu_wd(x, expert_ids, expert_weights, nullptr, Wg, Wu, Wd, wd_fmt, y, T, H, I, E,
                     top_k, stream, false);
}

zffn_status zffn_moe_swiglu_q4k_scaled(const void *x, const int32_t *expert_ids,
                                       const float *expert_weights, const float *down_scale,
                                       const void *Wg, const void *Wu, const void *Wd, int wd_fmt,
                                       float *y, int T, int H, int I, int E, int top_k,
                                       int accumulate, void *stream) {
    if (!expert_ids || !expert_weights) return invalid("expert_ids and expert_weights are required");
    return swiglu_wd(x, expert_ids, expert_weights, down_scale, Wg, Wu, Wd, wd_fmt, y, T, H, I, E,
                     top_k, stream, accumulate != 0);
}

zffn_status zffn_swiglu_q4k_wd(const void *x, const void *Wg, const void *Wu, const void *Wd,
                               int wd_fmt, float *y, int T, int H, int I, void *stream) {
    return zffn_moe_swiglu_q4k_wd(x, nullptr, nullptr, Wg, Wu, Wd, wd_fmt, y, T, H, I, 1, 1, stream);
}

zffn_status zffn_rmsnorm_bf16(const float *h, const float *gamma, float eps, void *x, int T, int H,
                              void *stream) {
    if (!h || !gamma || !x) return invalid("a pointer argument is NULL");
    if (T < 1) return invalid("T must be at least 1");
    if (H < 256 || H > 16384 || H % 256 != 0) return invalid("H must be a multiple of 256 in [256, 16384]");
    if (!(eps >= 0.0f) || eps > 1.0f) return invalid("eps must be in [0, 1]");
    if (!aligned16(h) || !aligned16(gamma) || !aligned16(x))
        return invalid("h, gamma and x must be 16-byte aligned");
    if (device_info().device < 0) return ZFFN_ERR_CUDA;
    return to_status(launch_rmsnorm_bf16(h, gamma, eps, static_cast<__nv_bfloat16 *>(x), T, H,
                                         (cudaStream_t)stream));
}

zffn_status zffn_swiglu_q4k_prenorm_residual(float *h, const float *gamma, float eps, const void *Wg,
                                             const void *Wu, const void *Wd, int T, int H, int I,
                                             void *stream) {
    if (!h || !gamma || !Wg || !Wu || !Wd) return invalid("a pointer argument is NULL");
    if (check_shape(T, H, I) != ZFFN_OK) return ZFFN_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || eps > 1.0f) return invalid("eps must be in [0, 1]");
    if (!aligned16(h) || !aligned16(gamma) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(Wd))
        return invalid("h, gamma, Wg, Wu and Wd must be 16-byte aligned");
    const DeviceInfo &di = device_info();
    if (di.device < 0) return ZFFN_ERR_CUDA;
    // the whole layout is reserved here, so that the block's own workspace
    // request below finds it large enough and never moves it
    const Layout L = layout_for(T, H, I, 1, 1);
    Workspace *w = nullptr;
    zffn_status st = ensure_workspace(L.total, &w);
    if (st != ZFFN_OK) return st;
    int mv_max;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        mv_max = g_matvec_max_t;
    }
    if (T == 1 && mv_max >= 1 && matvec_smem_bytes_prenorm(H, I) <= (size_t)di.max_smem_optin) {
        // one token: the normalisation runs inside the gate/up kernel, which
        // reads the residual row; the down kernel then adds into it
        MatvecArgs a{};
        a.norm_in = h;
        a.gamma = gamma;
        a.eps = eps;
        a.Wg = static_cast<const uint8_t *>(Wg);
        a.Wu = static_cast<const uint8_t *>(Wu);
        a.Wd = static_cast<const uint8_t *>(Wd);
        a.y = h;
        a.h = reinterpret_cast<float *>(static_cast<uint8_t *>(w->ptr) + L.h);
        a.err = di.err_word;
        a.T = 1; a.H = H; a.I = I; a.E = 1; a.k = 1;
        a.accumulate = true;
        return to_status(launch_ffn_matvec(a, (cudaStream_t)stream));
    }
    __nv_bfloat16 *xn = reinterpret_cast<__nv_bfloat16 *>(static_cast<uint8_t *>(w->ptr) + L.xn);
    cudaError_t e = launch_rmsnorm_bf16(h, gamma, eps, xn, T, H, (cudaStream_t)stream);
    if (e != cudaSuccess) return to_status(e);
    return swiglu_dense(xn, Wg, Wu, Wd, h, T, H, I, stream, true);
}

zffn_status zffn_moe_router_topk(const float *logits, int32_t *expert_ids, float *expert_weights,
                                 int T, int E, int top_k, void *stream) {
    if (!logits || !expert_ids || !expert_weights) return invalid("a pointer argument is NULL");
    if (T < 1 || E < 1 || E > 4096 || top_k < 1 || top_k > 64 || top_k > E)
        return invalid("T >= 1, E in [1, 4096] and top_k in [1, min(E, 64)] are required");
    if ((int64_t)T * E > ((int64_t)1 << 31) || (int64_t)T * top_k > (1 << 24))
        return invalid("T * E must not exceed 2^31 nor T * top_k 2^24");
    if ((reinterpret_cast<uintptr_t>(logits) & 3) || (reinterpret_cast<uintptr_t>(expert_ids) & 3) ||
        (reinterpret_cast<uintptr_t>(expert_weights) & 3))
        return invalid("logits, expert_ids and expert_weights must be 4-byte aligned");
    if (device_info().device < 0) return ZFFN_ERR_CUDA;
    return to_status(launch_moe_router(logits, T, E, top_k, expert_ids, expert_weights,
                                       (cudaStream_t)stream));
}

zffn_status zffn_reserve(int T_max, int H_max, int I_max, int E_max, int top_k_max) {
    if (T_max < 1 || H_max < 1 || I_max < 1 || E_max < 1 || top_k_max < 1)
        return invalid("every size must be at least 1");
    if (device_info().device < 0) return ZFFN_ERR_CUDA;
    const Layout L = layout_for(T_max, H_max, I_max, E_max, top_k_max);
    Workspace *w = nullptr;
    return ensure_workspace(L.total, &w);
}

int zffn_single_token_launches(int H, int I, int E, int top_k) {
    if (H < 1 || H > 65536 || I < 1 || I > 65536 || E < 1 || E > 65536 || top_k < 1 || top_k > 64) return -1;
    if (device_info().device < 0) return -1;
    int token_kernel;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        token_kernel = g_token_kernel;
    }
    return token_kernel == 0 && token_fused_fits_dims(H, I, top_k) ? 1 : 2;
}

size_t zffn_workspace_bytes(void) {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    return g_ws[dev].bytes;
}

void zffn_release(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    int prev = -1;
    cudaGetDevice(&prev);
    for (int d = 0; d < kMaxDevices; ++d) {
        if (g_ws[d].ptr) {
            cudaSetDevice(d);
            cudaFree(g_ws[d].ptr);
            g_ws[d] = Workspace{};
        }
    }
    if (prev >= 0) cudaSetDevice(prev);
}

zffn_status zffn_get_device_error(void *stream) {
    const DeviceInfo &di = device_info();
    if (di.device < 0) return ZFFN_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    int v = 0;
    if (cudaMemcpyAsync(&v, di.err_word, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return to_status(cudaErrorUnknown);
    if (cudaMemsetAsync(di.err_word, 0, sizeof(int), s) != cudaSuccess) return ZFFN_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return to_status(cudaErrorUnknown);
    if (v == ZFFN_ERR_TIMEOUT) {
        // a grid barrier that ran out leaves its count mid-count: start over
        std::lock_guard<std::mutex> lk(g_mu);
        Workspace &w = g_ws[di.device];
        if (w.ptr) {
            const Layout L = layout_for(1, 1, 1, 1, 1);
            if (cudaMemset(static_cast<uint8_t *>(w.ptr) + L.gbar, 0, sizeof(unsigned long long)) != cudaSuccess ||
                cudaDeviceSynchronize() != cudaSuccess)
                return to_status(cudaErrorUnknown);
        }
    }
    return v == 0 ? ZFFN_OK : (zffn_status)v;
}

const char *zffn_last_error(void) { return t_last_error; }

int zffn_set_option(int key, int value) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (key == ZFFN_OPT_MATVEC_MAX_T) {
        const int old = g_matvec_max_t;
        g_matvec_max_t = value < 0 ? 0 : value;
        return old;
    }
    if (key == ZFFN_OPT_MOE_KERNEL) {
        const int old = g_moe_kernel;
        g_moe_kernel = value < 0 || value > 2 ? 0 : value;
        return old;
    }
    if (key == ZFFN_OPT_TOKEN_KERNEL) {
        const int old = g_token_kernel;
        g_token_kernel = value == 1 ? 1 : 0;
        return old;
    }
    return -1;
}

zffn_status zffn_selftest_wait_timeout(int64_t budget_cycles, void *stream) {
    if (budget_cycles < 1) return invalid("budget_cycles must be at least 1");
    const DeviceInfo &di = device_info();
    if (di.device < 0) return ZFFN_ERR_CUDA;
    return to_status(launch_wait_timeout_selftest(budget_cycles, di.err_word, (cudaStream_t)stream));
}

}  // extern "C"

// ----------------------------------------------------------------------------
// Host pipeline: blocks over host buffers with the copies overlapped.
// ----------------------------------------------------------------------------
// Submission n uses slot n % depth: its x goes up on the upload stream, the
// block runs on the compute stream, y comes down on the download stream, and
// events order the three per slot (upload n waits for the block of n - depth
// to have read the slot's x; the block of n waits for upload n and for the
// download of n - depth to have emptied the slot's y).  So the copies of one
// submission overlap the blocks of its neighbours, and no call blocks the host
// except zffn_pipeline_sync.
struct zffn_pipeline {
    int device = -1;
    int T = 0, H = 0, I = 0, depth = 0;
    cudaStream_t up = nullptr, comp = nullptr, down = nullptr;
    void *x[ZFFN_PIPELINE_MAX_DEPTH] = {};
    float *y[ZFFN_PIPELINE_MAX_DEPTH] = {};
    cudaEvent_t in_done[ZFFN_PIPELINE_MAX_DEPTH] = {};
    cudaEvent_t comp_done[ZFFN_PIPELINE_MAX_DEPTH] = {};
    cudaEvent_t out_done[ZFFN_PIPELINE_MAX_DEPTH] = {};
    int64_t n = 0;
};

namespace {

void pipeline_free(zffn_pipeline *p) {
    if (!p) return;
    for (cudaStream_t s : {p->up, p->comp, p->down})
        if (s) cudaStreamSynchronize(s);
    for (int i = 0; i < ZFFN_PIPELINE_MAX_DEPTH; ++i) {
        if (p->x[i]) cudaFree(p->x[i]);
        if (p->y[i]) cudaFree(p->y[i]);
        if (p->in_done[i]) cudaEventDestroy(p->in_done[i]);
        if (p->comp_done[i]) cudaEventDestroy(p->comp_done[i]);
        if (p->out_done[i]) cudaEventDestroy(p->out_done[i]);
    }
    for (cudaStream_t s : {p->up, p->comp, p->down})
        if (s) cudaStreamDestroy(s);
    cudaGetLastError();
    delete p;
}

}  // namespace

extern "C" {

zffn_status zffn_pipeline_create(zffn_pipeline **out, int T, int H, int I, int depth) {
    if (!out) return invalid("out is NULL");
    *out = nullptr;
    if (check_shape(T, H, I) != ZFFN_OK) return ZFFN_ERR_INVALID_ARG;
    if (depth < 2 || depth > ZFFN_PIPELINE_MAX_DEPTH) return invalid("depth must be in [2, 4]");
    const DeviceInfo &di = device_info();
    if (di.device < 0) return ZFFN_ERR_CUDA;
    zffn_pipeline *p = new zffn_pipeline;
    p->device = di.device;
    p->T = T; p->H = H; p->I = I; p->depth = depth;
    cudaError_t e = cudaSuccess;
    for (cudaStream_t *s : {&p->up, &p->comp, &p->down})
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
    for (int i = 0; i < depth && e == cudaSuccess; ++i) {
        e = cudaMalloc(&p->x[i], (size_t)T * H * 2);
        if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void **>(&p->y[i]), (size_t)T * H * 4);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->in_done[i], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->comp_done[i], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->out_done[i], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) {
        const zffn_status st = e == cudaErrorMemoryAllocation ? ZFFN_ERR_NO_WORKSPACE : to_status(e);
        if (st == ZFFN_ERR_NO_WORKSPACE) set_last_error(cudaGetErrorString(e));
        pipeline_free(p);
        return st;
    }
    *out = p;
    return ZFFN_OK;
}

}  // extern "C"

namespace {

// One submission: upload, the block (`block(x_dev, y_dev, stream)`), download.
template <typename Block>
zffn_status pipeline_submit(zffn_pipeline *p, const void *x_host, float *y_host, Block block) {
    if (current_device() != p->device) return invalid("the pipeline belongs to another device");
    const int slot = (int)(p->n % p->depth);
    const size_t xb = (size_t)p->T * p->H * 2, yb = (size_t)p->T * p->H * 4;
    const bool reuse = p->n >= p->depth;
    cudaError_t e = cudaSuccess;
    if (reuse) e = cudaStreamWaitEvent(p->up, p->comp_done[slot], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(p->x[slot], x_host, xb, cudaMemcpyHostToDevice, p->up);
    if (e == cudaSuccess) e = cudaEventRecord(p->in_done[slot], p->up);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p->comp, p->in_done[slot], 0);
    if (e == cudaSuccess && reuse) e = cudaStreamWaitEvent(p->comp, p->out_done[slot], 0);
    if (e != cudaSuccess) return to_status(e);
    const zffn_status st = block(p->x[slot], p->y[slot], p->comp);
    if (st != ZFFN_OK) return st;
    e = cudaEventRecord(p->comp_done[slot], p->comp);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p->down, p->comp_done[slot], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(y_host, p->y[slot], yb, cudaMemcpyDeviceToHost, p->down);
    if (e == cudaSuccess) e = cudaEventRecord(p->out_done[slot], p->down);
    if (e != cudaSuccess) return to_status(e);
    ++p->n;
    return ZFFN_OK;
}

}  // namespace

extern "C" {

zffn_status zffn_pipeline_submit(zffn_pipeline *p, const void *x_host, const void *Wg, const void *Wu,
                                 const void *Wd, float *y_host) {
    if (!p || !x_host || !y_host || !Wg || !Wu || !Wd) return invalid("a pointer argument is NULL");
    return pipeline_submit(p, x_host, y_host, [&](void *x, float *y, cudaStream_t s) {
        return swiglu_dense(x, Wg, Wu, Wd, y, p->T, p->H, p->I, s, false);
    });
}

zffn_status zffn_pipeline_submit_moe(zffn_pipeline *p, const void *x_host, const int32_t *expert_ids,
                                     const float *expert_weights, const void *Wg, const void *Wu,
                                     const void *Wd, int E, int top_k, float *y_host) {
    if (!p || !x_host || !y_host || !expert_ids || !expert_weights || !Wg || !Wu || !Wd)
        return invalid("a pointer argument is NULL");
    return pipeline_submit(p, x_host, y_host, [&](void *x, float *y, cudaStream_t s) {
        return swiglu_moe(x, expert_ids, expert_weights, nullptr, Wg, Wu, Wd, y, p->T, p->H, p->I, E,
                          top_k, s, false);
    });
}

zffn_status zffn_pipeline_sync(zffn_pipeline *p) {
    if (!p) return invalid("the pipeline is NULL");
    for (cudaStream_t s : {p->up, p->comp, p->down}) {
        const cudaError_t e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return to_status(e);
    }
    return ZFFN_OK;
}

void zffn_pipeline_destroy(zffn_pipeline *p) { pipeline_free(p); }

}  // extern "C"
