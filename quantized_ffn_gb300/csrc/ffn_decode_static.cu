// ffn_decode_static.cu -- single-token dense block that allocates nothing.
//
// The regular entry points keep their scratch (the single-token path's
// intermediate strip) in a workspace that the library allocates with
// cudaMalloc on first use.  Some callers cannot allow
// that: a serving process whose own allocator has already claimed the whole
// device, a real-time loop that forbids allocation once it is running, or a
// caller that must never hit the implicit device synchronisation of
// cudaFree when a workspace grows.  This entry point runs the same kernel
// with its scratch in a fixed array compiled into the library instead.
//
// The array is a file-scope __device__ object: every GPU that loads the
// library holds it (64 KB) until the process exits.  Host code cannot
// use the array's name as a device address, so the first call on each device
// looks the address up with cudaGetSymbolAddress (with that device current)
// and caches it; that first call should therefore be made before any stream
// capture.  All calls share the one array, which keeps the last call's
// contents; calls whose launches overlap on the GPU race on the array.
#include <mutex>

#include "zffn_internal.cuh"

namespace zffn {

constexpr int kStaticMaxI = 16384;                 // largest intermediate width
constexpr size_t kStaticScratchFloats = kStaticMaxI;

static __device__ __align__(256) float g_static_scratch[kStaticScratchFloats];

namespace {
std::mutex g_static_mu;
float *g_static_ptr[64] = {};   // per device: address of g_static_scratch
}  // namespace

}  // namespace zffn

using namespace zffn;

extern "C" {

zffn_status zffn_swiglu_q4k_token_static(const void *x, const void *Wg, const void *Wu,
                                         const void *Wd, float *y, int H, int I, void *stream) {
    if (!x || !Wg || !Wu || !Wd || !y) {
        set_last_error("a pointer argument is NULL");
        return ZFFN_ERR_INVALID_ARG;
    }
    if (H < 256 || H > 16384 || H % 256 != 0 || I < 64 || I % 64 != 0) {
        set_last_error("H must be a multiple of 256 in [256, 16384] and I a multiple of 64");
        return ZFFN_ERR_INVALID_ARG;
    }
    if (I > kStaticMaxI) {
        set_last_error("I exceeds the static scratch limit of 16384");
        return ZFFN_ERR_INVALID_ARG;
    }
    const uintptr_t mask = 15;
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(Wg) |
         reinterpret_cast<uintptr_t>(Wu) | reinterpret_cast<uintptr_t>(Wd) |
         reinterpret_cast<uintptr_t>(y)) & mask) {
        set_last_error("pointers must be 16-byte aligned");
        return ZFFN_ERR_INVALID_ARG;
    }
    const DeviceInfo &di = device_info();
    if (di.device < 0) return ZFFN_ERR_CUDA;   // device_info recorded why
    if (di.device >= 64) {                     // g_static_ptr's size
        set_last_error("device index beyond the static scratch table");
        return ZFFN_ERR_CUDA;
    }
    if (matvec_smem_bytes(1, H, I, 1) > (size_t)di.max_smem_optin) {
        set_last_error("shape needs more shared memory than one block may use");
        return ZFFN_ERR_UNSUPPORTED;
    }
    float *scratch;
    {
        std::lock_guard<std::mutex> lk(g_static_mu);
        if (!g_static_ptr[di.device]) {
            void *p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
            if (e != cudaSuccess) {
                set_last_error(cudaGetErrorString(e));
                cudaGetLastError();
                return ZFFN_ERR_CUDA;
            }
            g_static_ptr[di.device] = static_cast<float *>(p);
        }
        scratch = g_static_ptr[di.device];
    }
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e;
    {
        MatvecArgs a{};
        a.x = static_cast<const __nv_bfloat16 *>(x);
        a.Wg = static_cast<const uint8_t *>(Wg);
        a.Wu = static_cast<const uint8_t *>(Wu);
        a.Wd = static_cast<const uint8_t *>(Wd);
        a.ids = nullptr;
        a.wts = nullptr;
        a.y = y;
        a.h = scratch;
        a.err = di.err_word;
        a.T = 1; a.H = H; a.I = I; a.E = 1; a.k = 1;
        a.accumulate = false;
        e = launch_ffn_matvec(a, s);
    }
    if (e != cudaSuccess) {
        set_last_error(cudaGetErrorString(e));
        cudaGetLastError();
        return ZFFN_ERR_CUDA;
    }
    return ZFFN_OK;
}

}  // extern "C"
