// moe_route.cu -- device-side preparation of a routed (mixture-of-experts)
// call: the chosen expert ids are read from the caller's device buffer and
// turned into per-expert row lists without any host readback ("Four
// bottlenecks, one CUDA backend...", section "Bottleneck 2 -- MoE decode was
// paying for its routing twice": the kernels index the right expert weights
// themselves).
//
//   route kernel (one block): count pairs per expert, exclusive scan into
//     row offsets, cut every expert's rows into tiles of at most tile_rows rows
//     (128, the prefill kernel's M, or 32, the grouped kernel's N), record for
//     each gathered row its token and routing weight.  Pairs with an id outside
//     [0, E) are dropped.
//   gather kernel: copy the x row of every gathered row into a contiguous
//     buffer, converted to fp16 (the tensor-core kernel's gate/up operand type),
//     so that the tensor-core kernel can load expert tiles with TMA.
#include "zffn_internal.cuh"

namespace zffn {

constexpr int kRouteThreads = 1024;

// Exclusive scan of v[0..n) in shared memory by one block; returns the total.
// Each thread sums a contiguous range, the per-thread sums are scanned with
// warp shuffles (within each warp, then across the warps' totals), and each
// thread writes the exclusive prefixes of its range.
__device__ int block_exclusive_scan(int *v, int n, int *scratch) {
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int lo = threadIdx.x * per, hi = min(n, lo + per);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = (blockDim.x + 31) >> 5;
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += v[i];
    // inclusive scan of the per-thread sums within the warp
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
    }
    if (lane == 31) scratch[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        // exclusive scan of the warp totals (at most 32 warps)
        const int wt = lane < nwarps ? scratch[lane] : 0;
        int winc = wt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, winc, o);
            if (lane >= o) winc += t;
        }
        scratch[lane] = winc - wt;                  // exclusive prefix of warp `lane`
        if (lane == 31) scratch[32] = winc;         // the total
    }
    __syncthreads();
    int run = scratch[warp] + inc - sum;            // exclusive prefix of this thread's range
    for (int i = lo; i < hi; ++i) {
        const int c = v[i];
        v[i] = run;
        run += c;
    }
    const int total = scratch[32];
    __syncthreads();
    return total;
}

__global__ void __launch_bounds__(kRouteThreads) moe_route_kernel(RouteArgs a) {
    extern __shared__ int sm[];
    int *cnt = sm;                       // [E]
    int *off = sm + a.E;                 // [E]
    int *tix = sm + 2 * a.E;             // [E]
    int *scratch = sm + 3 * a.E;         // [blockDim]
    const int P = a.T * a.k;
    // the gather kernel may be scheduled now; it waits for this grid's
    // completion before reading what this kernel writes
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < P; i += blockDim.x) {
        const int e = a.ids[i];
        if (e >= 0 && e < a.E) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
        off[e] = cnt[e];
        tix[e] = (cnt[e] + a.tile_rows - 1) / a.tile_rows;
        a.counts[e] = cnt[e];
    }
    __syncthreads();
    const int n_rows = block_exclusive_scan(off, a.E, scratch);
    const int n_tiles = block_exclusive_scan(tix, a.E, scratch);
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
        a.offsets[e] = off[e];
        const int nt = (cnt[e] + a.tile_rows - 1) / a.tile_rows;
        for (int t = 0; t < nt; ++t) {
            const int ti = tix[e] + t;
            if (ti < a.max_tiles)
                a.tiles[ti] = make_int4(off[e] + t * a.tile_rows, min(a.tile_rows, cnt[e] - t * a.tile_rows), e, 0);
        }
        cnt[e] = off[e];                 // becomes the fill cursor
    }
    if (threadIdx.x == 0) {
        a.offsets[a.E] = n_rows;
        *a.n_tiles = min(n_tiles, a.max_tiles);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < P; i += blockDim.x) {
        const int e = a.ids[i];
        if (e >= 0 && e < a.E) {
            const int pos = atomicAdd(&cnt[e], 1);
            a.row_token[pos] = i / a.k;
            a.row_weight[pos] = a.down_scale ? a.wts[i] * a.down_scale[e] : a.wts[i];
        }
    }
}

// Gathered rows of x (fp16, the tensor-core kernel's gate/up operand) and,
// in the same launch, y = 0 when the block is to overwrite y (its kernel adds
// its partial sums into y).
__global__ void __launch_bounds__(256) moe_gather_kernel(const __nv_bfloat16 *__restrict__ x,
                                                         const int *__restrict__ offsets, int E,
                                                         const int *__restrict__ row_token,
                                                         __half *__restrict__ x_perm,
                                                         int rows_cap, int H, float4 *__restrict__ y4,
                                                         int64_t ny4, float *ytail, int nytail) {
    // launched as a programmatic dependent of the routing kernel: wait for
    // its row lists (and for any earlier work on y) before touching memory
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int n_rows = min(offsets[E], rows_cap);
    const int vec = H / 8;   // 16-byte vectors per row
    for (int r = blockIdx.x; r < n_rows; r += gridDim.x) {
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (int64_t)row_token[r] * H);
        uint4 *dst = reinterpret_cast<uint4 *>(x_perm + (int64_t)r * H);
        for (int v = threadIdx.x; v < vec; v += blockDim.x) {
            // the tensor-core kernel takes its gate/up operand in fp16
            const uint4 w = src[v];
            dst[v] = make_uint4(bf16x2_to_f16x2_satfinite(w.x), bf16x2_to_f16x2_satfinite(w.y),
                                bf16x2_to_f16x2_satfinite(w.z), bf16x2_to_f16x2_satfinite(w.w));
        }
    }
    if (y4) {
        const int64_t stride = (int64_t)gridDim.x * blockDim.x;
        for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < ny4; i += stride)
            y4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (blockIdx.x == 0 && threadIdx.x < nytail) ytail[threadIdx.x] = 0.0f;
    }
}

// A dense block run as one expert on the grouped kernel: consecutive groups of
// `rows` tokens, weight 1.
__global__ void __launch_bounds__(256) dense_groups_kernel(int T, int rows, int4 *tiles, int *n_tiles,
                                                           int *row_token, float *row_weight) {
    const int n = (T + rows - 1) / rows;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < T; i += gridDim.x * blockDim.x) {
        row_token[i] = i;
        row_weight[i] = 1.0f;
        if (i % rows == 0) tiles[i / rows] = make_int4(i, min(rows, T - i), 0, 0);
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) *n_tiles = n;
}

cudaError_t launch_dense_groups(int T, int rows, int4 *tiles, int *n_tiles, int *row_token, float *row_weight,
                                cudaStream_t s) {
    int grid = (T + 255) / 256;
    if (grid > device_info().num_sms * 4) grid = device_info().num_sms * 4;
    dense_groups_kernel<<<grid, 256, 0, s>>>(T, rows, tiles, n_tiles, row_token, row_weight);
    return cudaGetLastError();
}

cudaError_t launch_moe_route(const RouteArgs &a, cudaStream_t s) {
    const size_t smem = (size_t)(3 * a.E + kRouteThreads) * sizeof(int);
    if (smem > 48 * 1024) {
        cudaError_t e = ensure_dynamic_smem((const void *)moe_route_kernel, smem);
        if (e != cudaSuccess) return e;
    }
    moe_route_kernel<<<1, kRouteThreads, smem, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int P = a.T * a.k;
    int grid = P < device_info().num_sms * 8 ? P : device_info().num_sms * 8;
    if (grid < 1) grid = 1;
    const int64_t ny4 = a.y_zero ? a.ny / 4 : 0;
    // a programmatic dependent of the routing kernel: its launch overlaps
    // that kernel, and it waits for its completion itself
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, moe_gather_kernel, a.x, (const int *)a.offsets, a.E, (const int *)a.row_token,
                              a.x_perm, P, a.H, reinterpret_cast<float4 *>(a.y_zero), ny4,
                              a.y_zero ? a.y_zero + 4 * ny4 : (float *)nullptr,
                              a.y_zero ? (int)(a.ny - 4 * ny4) : 0);
}

// ---------------------------------------------------------------------------
// Bounded-wait self test: one block waits on an mbarrier whose expected
// arrival never comes; the wait gives up after the budget and records
// ZFFN_ERR_TIMEOUT, and the kernel returns normally.
// ---------------------------------------------------------------------------
__global__ void wait_timeout_selftest_kernel(long long budget, int *err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 2);          // two arrivals expected ...
        fence_mbarrier_init();
        mbar_arrive(&bar);           // ... and only one ever happens
        mbar_wait(&bar, 0, nullptr, err, budget);
    }
    __syncthreads();
}

cudaError_t launch_wait_timeout_selftest(int64_t budget_cycles, int *err, cudaStream_t s) {
    wait_timeout_selftest_kernel<<<1, 32, 0, s>>>((long long)budget_cycles, err);
    return cudaGetLastError();
}

}  // namespace zffn
