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
// ahead > 0: thread 0 also warms L2 with the CTA's input slices of row + ahead (bulk prefetches of the residual
// and x, or of the residual and every partial), the row a later wave runs on this slot, so that its loads meet L2
// while this wave sits in its reduction and epilogue.
template <int VPT, int EP, bool ALLRED, int CL>
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
    if (ahead > 0 && row + ahead < p.rows && threadIdx.x == 0) {
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
        norm_row_slice<VPT, EP, ALLRED, CL>(p, row, rank, ctas_per_row, begin, end, sm, pslices, slice, smem_addr(&pbar));
    } else {
        norm_row_slice<VPT, EP, ALLRED, CL>(p, row, rank, ctas_per_row, begin, end, sm);
    }
    pdl_leave(order);
}

// Per device and partial-sum kernel variant (epilogue x row in one CTA or a cluster): the id of the context in
// which its preferred carveout, the largest shared-memory share, was last requested, so that shared memory
// (n_partials x slice vectors per CTA) rather than the L1 share bounds the resident CTAs. A kernel attribute
// belongs to a context; with no context id (0) every launch requests it.
std::atomic<unsigned long long> g_partials_carveout_ctx[kMaxCachedDevices][8];

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

// Wave-ahead distance of a launch of more rows than fit on the GPU at once (R = SMs x resident CTAs per SM /
// CTAs per row): R / 2 rows for the plain norm, R / 8 for the all-reduce half, whose bulk copies of the partials
// already keep many bytes in flight and whose rows are nine or more row-sized reads (a longer distance evicts
// rows before they are used). Measured on GB300 over 0 to R (CUDA events around back-to-back launches, inputs
// above 3x L2): the plain norm peaks between 3R/8 and 3R/4 (NVFP4 T 2048, H 16384: 36.65 -> 35.65 us; static
// FP8 T 1000, H 16384: 20.10 -> 19.28; bf16 T 2048, H 4096: 12.32 -> 11.56), the all-reduce half at R / 8 (k 8,
// T 2048, H 16384, static FP8: 124.0 -> 119.6 us) and falls below no warming past R / 2.
int wave_ahead(const NormParams& p, const RowPlan& plan, const void* kern, size_t smem) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    const int64_t resident = int64_t{sms} * resident_ctas_per_sm(dev, kern, plan.threads, smem) / plan.ctas_per_row;
    if (resident <= 0 || p.rows <= resident) return 0;
    return static_cast<int>(p.n_partials > 0 ? resident / 8 : resident / 2);
}

template <int EP>
cudaError_t launch_ep(const NormParams& p, const RowPlan& plan, cudaStream_t s) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    void (*kern)(NormParams, int, int, int, int, int) = nullptr;
    const bool cl = plan.ctas_per_row > 1;
    if (p.n_partials > 0) {
        if (plan.vpt != 1) return cudaErrorInvalidValue;
        kern = cl ? add_rmsnorm_kernel<1, EP, true, kRowInCluster> : add_rmsnorm_kernel<1, EP, true, kRowInCta>;
    } else {
        switch (plan.vpt) {
            case 1: kern = cl ? add_rmsnorm_kernel<1, EP, false, kRowInCluster> : add_rmsnorm_kernel<1, EP, false, kRowInCta>; break;
            case 2: kern = cl ? add_rmsnorm_kernel<2, EP, false, kRowInCluster> : add_rmsnorm_kernel<2, EP, false, kRowInCta>; break;
            case 4: kern = cl ? add_rmsnorm_kernel<4, EP, false, kRowInCluster> : add_rmsnorm_kernel<4, EP, false, kRowInCta>; break;
            case 8: kern = cl ? add_rmsnorm_kernel<8, EP, false, kRowInCluster> : add_rmsnorm_kernel<8, EP, false, kRowInCta>; break;
            default: return cudaErrorInvalidValue;
        }
    }
    fill_launch(cfg, attr, p.rows, plan.ctas_per_row, plan.threads, plan.ctas_per_row, s);
    if (p.n_partials > 0) {
        const cudaError_t ce = prefer_shared_carveout(reinterpret_cast<const void*>(kern), EP * 2 + (cl ? 1 : 0));
        if (ce != cudaSuccess) return ce;
        const size_t smem = static_cast<size_t>(p.n_partials) * static_cast<size_t>(plan.slice) * 16;
        if (smem > 48 * 1024) {   // above the default dynamic shared-memory limit: opt in (a kernel attribute)
            const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       static_cast<int>(smem));
            if (e != cudaSuccess) return e;
        }
        cfg.dynamicSmemBytes = smem;
    }
    const int ahead = wave_ahead(p, plan, reinterpret_cast<const void*>(kern), cfg.dynamicSmemBytes);
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
