// Fused SwiGLU over the stacked gate_up projection (+ FP8 E4M3 or NVFP4 epilogue).
//
// Definition ("TensorRT-LLM: Compiling Inference Engines Ahead of Time", "Fusing operations, measured"):
// gate and up are the two halves of one stacked projection row, combined per element as
// g / (1 + exp(-g)) * up by a fused kernel, so the [T, I] activation is not written out and read back.
// The FP8 variant follows the SiLU-plus-quantisation fusion of "Introduction to torch.compile and How It
// Works with vLLM" (section 3, custom compiler passes): the activation leaves as E4M3 codes for the next
// GEMM in the same pass.
//
// bf16, static-scale and NVFP4 variants are pure streams (no row reduction; NVFP4's 16-element block maximum
// is one shuffle between neighbouring lanes): each CTA owns a slice of one row.
// The dynamic per-token variant keeps the slice's fp32 products in registers, reduces max |h| over the row
// (warp shuffles, shared memory, and distributed shared memory across the row's cluster), then quantises
// from the registers, so the activation crosses HBM exactly once.
#include "swiglu_impl.cuh"

namespace mbd {

namespace {

template <int VPT, int EP>
__global__ void __launch_bounds__(512, VPT <= 2 ? 4 : 1) swiglu_kernel(const __grid_constant__ SwigluParams p, int ctas_per_row, int slice, int prefetch,
                                                                   int ahead) {
    __shared__ SwigluSmem sm;
    const int64_t row = launch_row();
    if (row >= p.rows) return;   // past the last row (the whole cluster shares the row)
    const int rank = static_cast<int>(blockIdx.x);
    const int begin = rank * slice;
    const int end = min(begin + slice, p.nvec);
    pdl_trigger();
    if (prefetch) swiglu_prefetch<VPT>(p, row, begin, end);
    pdl_wait();
    // The row a later wave will run here is fetched into L2 now, so that its loads meet L2 instead of HBM;
    // the bytes come from HBM once either way (the rows in flight plus those ahead fit L2 many times over).
    // Two bulk prefetches (gate and up slices) from one thread.
    if (ahead > 0 && row + ahead < p.rows && threadIdx.x == 0) {
        const uint4* gr = static_cast<const uint4*>(p.gate_up) + (row + ahead) * (int64_t)p.nvec * 2 + begin;
        const uint32_t bytes = static_cast<uint32_t>(end - begin) * 16u;
        prefetch_l2_bulk(gr, bytes);
        prefetch_l2_bulk(gr + p.nvec, bytes);
    }
    swiglu_row_slice<VPT, EP>(p, row, rank, ctas_per_row, begin, end, sm);
}

template <int EP>
cudaError_t launch_ep(const SwigluParams& p, const RowPlan& plan, cudaStream_t s) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    const int cluster = EP == kFp8Dynamic ? plan.ctas_per_row : 1;
    void (*kern)(SwigluParams, int, int, int, int) = nullptr;
    switch (plan.vpt) {
        case 1: kern = swiglu_kernel<1, EP>; break;
        case 2: kern = swiglu_kernel<2, EP>; break;
        case 4: kern = swiglu_kernel<4, EP>; break;
        case 8: kern = swiglu_kernel<8, EP>; break;
        default: return cudaErrorInvalidValue;
    }
    fill_launch(cfg, attr, p.rows, plan.ctas_per_row, plan.threads, cluster, s);
    return cudaLaunchKernelEx(&cfg, kern, p, plan.ctas_per_row, plan.slice, plan.prefetch, plan.ahead);
}

}  // namespace

cudaError_t device_error_flags_swiglu(unsigned int* flags, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_device_error_flags, sizeof(unsigned int));
    if (e == cudaSuccess && clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error_flags, &zero, sizeof(unsigned int));
    }
    return e;
}

cudaError_t launch_swiglu(const SwigluParams& p, Epilogue ep, const RowPlan& plan, cudaStream_t s) {
    switch (ep) {
        case kBf16: return launch_ep<kBf16>(p, plan, s);
        case kFp8Static: return launch_ep<kFp8Static>(p, plan, s);
        case kFp8Dynamic: return launch_ep<kFp8Dynamic>(p, plan, s);
        case kNvfp4: return launch_ep<kNvfp4>(p, plan, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace mbd
