// Fused residual add + RMSNorm (+ FP8 E4M3 or NVFP4 epilogue).
//
// Definition ("TensorRT-LLM: Compiling Inference Engines Ahead of Time", "Fusing operations, measured"):
// RMSNorm is an eight-step chain (float cast, square, mean, epsilon, reciprocal square root, scaling,
// cast back, weight), and TensorRT-LLM runs the residual addition inside the normalisation kernel. Here
// that whole chain is one pass over HBM: each row is read once (x, residual), the rounded
// sum is written back as the new residual, and the normalised row leaves as bf16 or as E4M3 codes
// (the Quantize half of the fusions listed in "Introduction to torch.compile and How It Works with
// vLLM", section 4).
//
// Data flow per row slice: 16-byte loads of x and residual into registers -> s = bf16(x + r) (kept packed)
// -> residual store -> sum of s^2 -> CTA (+cluster) reduction -> inv = 1/sqrt(mean + eps) -> weight loads
// -> v = (w * s) * inv -> bf16 store, E4M3 codes with a static scale, or NVFP4 (E2M1 codes under an E4M3
// scale per 16 elements and the fp32 tensor scale, the Blackwell 4-bit format described in the TensorRT-LLM
// walkthrough, Part V, quantization co-designed with the hardware). The dynamic per-token variant
// reduces the sum of squares and max |w * s| together (the scale is max |w * s| * inv / 448), then stores
// the codes from registers.
#include <atomic>
#include <mutex>
#include <vector>

#include "norm_impl.cuh"

namespace mbd {

namespace {

// The partial-sum form brings the CTA's slices of the partials into shared memory with bulk copies (one thread
// issues them; dynamic shared memory, n_partials x slice vectors) and asks for three 512-thread CTAs' worth of
// registers per SM: registers hold one partial vector at a time, not all of them.
// AHEAD: thread 0 also warms L2 with the CTA's input slices of row + ahead (bulk prefetches of the residual and
// x, or of the residual and every partial), the row a later wave runs on this slot, so that its loads meet L2
// while this wave sits in its reduction and epilogue. A compile-time choice: the branch alone, never taken, cost
// single-wave launches 0.1 to 0.4 us (static FP8, H 16384, T 16: 2.52 -> 2.90 us).
template <int VPT, int EP, bool ALLRED, int CL, bool AHEAD>
__global__ void __launch_bounds__(512, ALLRED ? 3 : 1) add_rmsnorm_kernel(const __grid_constant__ NormParams p, int ctas_per_row, int slice,
                                                                        int prefetch, int ahead, int order) {
    extern __shared__ __align__(16) uint4 pslices[];   // all-reduce half: partial k's slice at [k * slice, ...)
    __shared__ NormSmem sm;
    __shared__ unsigned long long pbar;
    const int64_t row = launch_row();
    if (row >= p.rows) return;   // past the last row (the whole cluster shares the row)
    const int rank = static_cast<int>(blockIdx.x);
    const int begin = rank * slice;
    const int end = min(begin + slice, p.nvec);
    pdl_enter_trigger(order);
    if constexpr (ALLRED) {
        if (threadIdx.x == 0) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&pbar)) : "memory");
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
    }
    if (prefetch) norm_prefetch<VPT, ALLRED>(p, row, begin, end);
    pdl_enter_wait(order);
    if (AHEAD && row + ahead < p.rows && threadIdx.x == 0) {
        const uint32_t bytes = static_cast<uint32_t>(end - begin) * 16u;
        const int64_t at = (row + ahead) * static_cast<int64_t>(p.nvec) + begin;
        prefetch_l2_bulk(static_cast<const uint4*>(p.residual) + at, bytes);
        if constexpr (ALLRED) {
            for (int k = 0; k < p.n_partials; ++k) prefetch_l2_bulk(static_cast<const uint4*>(p.partials[k]) + at, bytes);
        } else {
            prefetch_l2_bulk(static_cast<const uint4*>(p.x) + at, bytes);
        }
    }
    if constexpr (ALLRED) {
        if (threadIdx.x == 0) load_partials_bulk(p, row, begin, end - begin, slice, pslices, smem_addr(&pbar));
        norm_row_slice<VPT, EP, ALLRED, CL, true>(p, row, rank, ctas_per_row, begin, end, sm, pslices, slice,
                                                 smem_addr(&pbar));
    } else {
        norm_row_slice<VPT, EP, ALLRED, CL, true>(p, row, rank, ctas_per_row, begin, end, sm);
    }
    pdl_leave(order);
}

// Per device and partial-sum kernel variant (epilogue x row in one CTA or a cluster x warming): the id of the
// context in which its preferred carveout, the largest shared-memory share, was last requested, so that shared
// memory (n_partials x slice vectors per CTA) rather than the L1 share bounds the resident CTAs. A kernel attribute
// belongs to a context; with no context id (0) every launch requests it.
std::atomic<unsigned long long> g_partials_carveout_ctx[kMaxCachedDevices][16];

cudaError_t prefer_shared_carveout(const void* kern, int variant) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long ctx = current_context_id();
    if (dev < 0 || dev >= kMaxCachedDevices || ctx == 0 ||
        g_partials_carveout_ctx[dev][variant].load(std::memory_order_acquire) != ctx) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 static_cast<int>(cudaSharedmemCarveoutMaxShared));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kMaxCachedDevices) g_partials_carveout_ctx[dev][variant].store(ctx, std::memory_order_release);
    }
    return cudaSuccess;
}

// Resident CTAs per SM of a kernel at a block size and dynamic shared-memory size (the occupancy calculator,
// which also sees the kernel's carveout preference), cached per device, context, kernel and launch shape. 0 when
// the calculator fails (no warming then; its error is cleared).
struct ResidentKey {
    int dev;
    unsigned long long ctx;
    const void* kern;
    int threads;
    size_t smem;
};
std::mutex g_resident_mu;
std::vector<std::pair<ResidentKey, int>> g_resident;
constexpr size_t kMaxResidentEntries = 256;

int resident_ctas_per_sm(int dev, const void* kern, int threads, size_t smem) {
    const unsigned long long ctx = current_context_id();
    {
        std::lock_guard<std::mutex> lock(g_resident_mu);
        for (const auto& e : g_resident)
            if (e.first.dev == dev && e.first.ctx == ctx && e.first.kern == kern && e.first.threads == threads &&
                e.first.smem == smem)
                return e.second;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    if (ctx != 0) {
        std::lock_guard<std::mutex> lock(g_resident_mu);
        if (g_resident.size() >= kMaxResidentEntries) g_resident.clear();
        g_resident.push_back({ResidentKey{dev, ctx, kern, threads, smem}, n});
    }
    return n;
}

// Wave-ahead distance of a launch (R = SMs x resident CTAs per SM / CTAs per row, the rows that fit on the GPU at
// once): R / 2 rows for the plain norm from 2R rows on with the bf16 epilogue and from 4R rows on with the FP8 and
// NVFP4 ones; R / 8 for the all-reduce half from R rows on, whose bulk copies of the partials already keep many
// bytes in flight and whose rows are nine or more row-sized reads (a longer distance evicts rows before they are
// used). Measured on GB300 (CUDA-graph replay, inputs above 3x L2, each shape with and without): the distance is
// best between 3R/8 and 3R/4 for the plain norm, at R / 8 for the all-reduce half, and costs time past R; the
// warming pays from about 4R rows with the quantising epilogues (static FP8, H 16384: T 1000 +0.3%, T 3000 -6%,
// T 8192 -9%; NVFP4, H 16384: T 1000 +3.5%, T 2048 -1.6%, T 8192 -11%) and from about 2R with bf16 (H 4096:
// T 3000 -3%, T 4096 -2.5%; H 5120: T 2048 -2%); the all-reduce half, k 8, T 2048, H 16384, static FP8: 127.5 ->
// 123.6 us (the bench's per-unit breakdown).
int wave_ahead(const NormParams& p, const RowPlan& plan, const void* kern, size_t smem, int min_waves) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    const int64_t resident = int64_t{sms} * resident_ctas_per_sm(dev, kern, plan.threads, smem) / plan.ctas_per_row;
    if (resident <= 0 || p.rows < resident * min_waves || p.rows <= resident) return 0;
    return static_cast<int>(p.n_partials > 0 ? resident / 8 : resident / 2);
}

using NormKernel = void (*)(NormParams, int, int, int, int, int);

// The kernel of a plan: the partial-sum form (one vector per thread) or the plain one, with or without warming.
template <int EP, bool AHEAD>
NormKernel norm_kernel(const NormParams& p, const RowPlan& plan) {
    const bool cl = plan.ctas_per_row > 1;
    if (p.n_partials > 0) {
        if (plan.vpt != 1) return nullptr;
        return cl ? add_rmsnorm_kernel<1, EP, true, kRowInCluster, AHEAD> : add_rmsnorm_kernel<1, EP, true, kRowInCta, AHEAD>;
    }
    switch (plan.vpt) {
        case 1: return cl ? add_rmsnorm_kernel<1, EP, false, kRowInCluster, AHEAD> : add_rmsnorm_kernel<1, EP, false, kRowInCta, AHEAD>;
        case 2: return cl ? add_rmsnorm_kernel<2, EP, false, kRowInCluster, AHEAD> : add_rmsnorm_kernel<2, EP, false, kRowInCta, AHEAD>;
        case 4: return cl ? add_rmsnorm_kernel<4, EP, false, kRowInCluster, AHEAD> : add_rmsnorm_kernel<4, EP, false, kRowInCta, AHEAD>;
        case 8: return cl ? add_rmsnorm_kernel<8, EP, false, kRowInCluster, AHEAD> : add_rmsnorm_kernel<8, EP, false, kRowInCta, AHEAD>;
        default: return nullptr;
    }
}

// The partial-sum kernels' attributes: the carveout (above) and, above the default 48 KB, the opt-in to the
// CTA's dynamic shared memory (n_partials x slice vectors).
cudaError_t prepare_partials_kernel(NormKernel kern, int variant, size_t smem) {
    const cudaError_t ce = prefer_shared_carveout(reinterpret_cast<const void*>(kern), variant);
    if (ce != cudaSuccess) return ce;
    if (smem > 48 * 1024)
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    return cudaSuccess;
}

template <int EP>
cudaError_t launch_ep(const NormParams& p, const RowPlan& plan, cudaStream_t s) {
    const bool partials = p.n_partials > 0;
    const int variant = EP * 2 + (plan.ctas_per_row > 1 ? 1 : 0);
    const size_t smem = partials ? static_cast<size_t>(p.n_partials) * static_cast<size_t>(plan.slice) * 16 : 0;
    // the warming form where the launch has more rows than fit at once (its residency decides), else the plain one
    NormKernel kern = norm_kernel<EP, true>(p, plan);
    if (kern == nullptr) return cudaErrorInvalidValue;
    if (partials) {
        const cudaError_t e = prepare_partials_kernel(kern, variant + 8, smem);
        if (e != cudaSuccess) return e;
    }
    const int min_waves = partials ? 1 : (EP == kBf16 ? 2 : 4);
    const int ahead = wave_ahead(p, plan, reinterpret_cast<const void*>(kern), smem, min_waves);
    if (ahead == 0) {
        kern = norm_kernel<EP, false>(p, plan);
        if (partials) {
            const cudaError_t e = prepare_partials_kernel(kern, variant, smem);
            if (e != cudaSuccess) return e;
        }
    }
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    fill_launch(cfg, attr, p.rows, plan.ctas_per_row, plan.threads, plan.ctas_per_row, s);
    cfg.dynamicSmemBytes = smem;
    return cudaLaunchKernelEx(&cfg, kern, p, plan.ctas_per_row, plan.slice, plan.prefetch, ahead, plan.order);
}

}  // namespace

cudaError_t device_error_flags_norm(unsigned int* flags, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_device_error_flags, sizeof(unsigned int));
    if (e == cudaSuccess && clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error_flags, &zero, sizeof(unsigned int));
    }
    return e;
}

cudaError_t launch_add_rmsnorm(const NormParams& p, Epilogue ep, const RowPlan& plan, cudaStream_t s) {
    switch (ep) {
        case kBf16: return launch_ep<kBf16>(p, plan, s);
        case kFp8Static: return launch_ep<kFp8Static>(p, plan, s);
        case kFp8Dynamic: return launch_ep<kFp8Dynamic>(p, plan, s);
        case kNvfp4: return launch_ep<kNvfp4>(p, plan, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace mbd
