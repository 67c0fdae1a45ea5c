// Fused SwiGLU over the stacked gate_up projection (+ FP8 E4M3 epilogue).
//
// Definition ("TensorRT-LLM: Compiling Inference Engines Ahead of Time", "Fusing operations, measured"):
// the gated MLP runs one gate_up matmul whose row holds gate in its first half and up in its second half,
// then a swiglu kernel that computes g / (1 + exp(-g)) * up per element, so the [T, I] intermediate is
// never written and re-read. The FP8 variant is the Quantize(SiLU(x)) fusion of "Introduction to
// torch.compile and How It Works with vLLM" (section 3, custom compiler passes): the activation is
// quantised to E4M3 for the next GEMM inside the same pass.
//
// bf16 and static-scale variants are pure streams (no reduction): each CTA owns a slice of one row.
// The dynamic per-token variant keeps the slice's fp32 products in registers, reduces max |h| over the row
// (warp shuffles, shared memory, and distributed shared memory across the row's cluster), then quantises
// from the registers, so the activation crosses HBM exactly once.
#include "common.cuh"
#include "launch.h"

namespace mbd {

namespace {

__device__ __forceinline__ float silu_times(float g, float u) { return g / (1.0f + expf(-g)) * u; }

template <int VPT, int EP>
__global__ void __launch_bounds__(512) swiglu_kernel(SwigluParams p, int ctas_per_row, int slice) {
    __shared__ float red_max[32];
    __shared__ float cl_slot[1];

    const int64_t row = blockIdx.x / ctas_per_row;
    const int rank = blockIdx.x - static_cast<int>(row * ctas_per_row);
    const int begin = rank * slice;
    const int end = min(begin + slice, p.nvec);

    const uint4* gr = static_cast<const uint4*>(p.gate_up) + row * (int64_t)p.nvec * 2;
    const uint4* ur = gr + p.nvec;

    uint4 gv[VPT], uv[VPT];
    bool live[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int c = begin + threadIdx.x + i * blockDim.x;
        live[i] = c < end;
        if (live[i]) {
            gv[i] = load_stream(gr + c);
            uv[i] = load_stream(ur + c);
        }
    }

    if constexpr (EP == kBf16) {
        uint4* outr = static_cast<uint4*>(p.out) + row * (int64_t)p.nvec;
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            if (!live[i]) continue;
            const uint32_t* gw = reinterpret_cast<const uint32_t*>(&gv[i]);
            const uint32_t* uw = reinterpret_cast<const uint32_t*>(&uv[i]);
            uint4 o;
            uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                ow[k] = pack_bf16x2(silu_times(bf16_lo(gw[k]), bf16_lo(uw[k])),
                                    silu_times(bf16_hi(gw[k]), bf16_hi(uw[k])));
            store_stream(outr + (begin + threadIdx.x + i * blockDim.x), o);
        }
    } else {
        uint2* outr = reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.out) + row * (int64_t)p.nvec * 8);
        float h[VPT][8];
        float qmul;
        if constexpr (EP == kFp8Static) {
            const float sc = __ldg(p.scale);
            qmul = sc > 0.0f ? 1.0f / sc : 0.0f;
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            if (!live[i]) continue;
            const uint32_t* gw = reinterpret_cast<const uint32_t*>(&gv[i]);
            const uint32_t* uw = reinterpret_cast<const uint32_t*>(&uv[i]);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                h[i][2 * k] = silu_times(bf16_lo(gw[k]), bf16_lo(uw[k]));
                h[i][2 * k + 1] = silu_times(bf16_hi(gw[k]), bf16_hi(uw[k]));
                if constexpr (EP == kFp8Dynamic)
                    amax = fmaxf(amax, fmaxf(fabsf(h[i][2 * k]), fabsf(h[i][2 * k + 1])));
            }
        }
        if constexpr (EP == kFp8Dynamic) {
            amax = cta_allreduce(amax, red_max, MaxOp{});
            amax = cluster_allreduce(amax, &cl_slot[0], ctas_per_row, MaxOp{});
            const float sc = amax / 448.0f;
            qmul = sc > 0.0f ? 1.0f / sc : 0.0f;
            if (rank == 0 && threadIdx.x == 0) p.scale[row] = sc;
        }
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            if (!live[i]) continue;
            uint2 q;
            q.x = pack_e4m3x4(h[i][0] * qmul, h[i][1] * qmul, h[i][2] * qmul, h[i][3] * qmul);
            q.y = pack_e4m3x4(h[i][4] * qmul, h[i][5] * qmul, h[i][6] * qmul, h[i][7] * qmul);
            store_stream(outr + (begin + threadIdx.x + i * blockDim.x), q);
        }
        if constexpr (EP == kFp8Dynamic) cluster_sync_if(ctas_per_row);
    }
}

template <int EP>
cudaError_t launch_ep(const SwigluParams& p, const RowPlan& plan, cudaStream_t s) {
    void (*kern)(SwigluParams, int, int) = nullptr;
    switch (plan.vpt) {
        case 1: kern = swiglu_kernel<1, EP>; break;
        case 2: kern = swiglu_kernel<2, EP>; break;
        case 4: kern = swiglu_kernel<4, EP>; break;
        case 8: kern = swiglu_kernel<8, EP>; break;
        default: return cudaErrorInvalidValue;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.rows * plan.ctas_per_row), 1, 1);
    cfg.blockDim = dim3(plan.threads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = plan.ctas_per_row;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (EP == kFp8Dynamic && plan.ctas_per_row > 1) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p, plan.ctas_per_row, plan.slice);
}

}  // namespace

cudaError_t launch_swiglu(const SwigluParams& p, Epilogue ep, const RowPlan& plan, cudaStream_t s) {
    switch (ep) {
        case kBf16: return launch_ep<kBf16>(p, plan, s);
        case kFp8Static: return launch_ep<kFp8Static>(p, plan, s);
        case kFp8Dynamic: return launch_ep<kFp8Dynamic>(p, plan, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace mbd
