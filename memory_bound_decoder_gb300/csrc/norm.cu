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
#include "norm_impl.cuh"

namespace mbd {

namespace {

// The partial-sum form asks for two 512-thread CTAs per SM (<= 64 registers): its eight loads in flight
// per vector would otherwise leave one CTA, a quarter of the SM's warps.
template <int VPT, int EP, bool ALLRED, int CL>
__global__ void __launch_bounds__(512, ALLRED ? 2 : 1) add_rmsnorm_kernel(const __grid_constant__ NormParams p, int ctas_per_row, int slice,
                                                                        int prefetch, int order) {
    __shared__ NormSmem sm;
    const int64_t row = launch_row();
    if (row >= p.rows) return;   // past the last row (the whole cluster shares the row)
    const int rank = static_cast<int>(blockIdx.x);
    const int begin = rank * slice;
    const int end = min(begin + slice, p.nvec);
    pdl_enter_trigger(order);
    if (prefetch) norm_prefetch<VPT, ALLRED>(p, row, begin, end);
    pdl_enter_wait(order);
    norm_row_slice<VPT, EP, ALLRED, CL>(p, row, rank, ctas_per_row, begin, end, sm);
    pdl_leave(order);
}

template <int EP>
cudaError_t launch_ep(const NormParams& p, const RowPlan& plan, cudaStream_t s) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    void (*kern)(NormParams, int, int, int, int) = nullptr;
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
    return cudaLaunchKernelEx(&cfg, kern, p, plan.ctas_per_row, plan.slice, plan.prefetch, plan.order);
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
