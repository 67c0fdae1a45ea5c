// Fused residual add + RMSNorm (+ FP8 E4M3 epilogue).
//
// Definition ("TensorRT-LLM: Compiling Inference Engines Ahead of Time", "Fusing operations, measured"):
// RMSNorm is the chain cast-to-float, square, mean, add epsilon, reciprocal square root, multiply,
// cast back, multiply by the weight, and TensorRT-LLM's module adds the residual and normalises in one
// kernel. Here that whole chain is one pass over HBM: each row is read once (x, residual), the rounded
// sum is written back as the new residual, and the normalised row leaves as bf16 or as E4M3 codes
// (the Quantize half of the fusions listed in "Introduction to torch.compile and How It Works with
// vLLM", section 4).
//
// Data flow per row slice: 16-byte loads of x and residual into registers -> s = bf16(x + r) (kept packed)
// -> residual store -> sum of s^2 -> CTA (+cluster) reduction -> inv = 1/sqrt(mean + eps) -> weight loads
// -> v = s * inv * w -> bf16 store, or E4M3 codes with a static scale, or (dynamic) a second reduction of
// max |v| followed by recomputing v and storing the codes.
#include "common.cuh"
#include "launch.h"

namespace mbd {

namespace {

template <int VPT, int EP>
__global__ void __launch_bounds__(512) add_rmsnorm_kernel(NormParams p, int ctas_per_row, int slice) {
    __shared__ float red_sum[32];
    __shared__ float red_max[32];
    __shared__ float cl_slot[2];

    const int64_t row = blockIdx.x / ctas_per_row;
    const int rank = blockIdx.x - static_cast<int>(row * ctas_per_row);
    const int begin = rank * slice;
    const int end = min(begin + slice, p.nvec);

    const uint4* xr = static_cast<const uint4*>(p.x) + row * p.nvec;
    uint4* rr = static_cast<uint4*>(p.residual) + row * p.nvec;
    const uint4* wr = static_cast<const uint4*>(p.weight);

    uint4 sv[VPT];
    bool live[VPT];
    {
        uint4 xv[VPT], rv[VPT];
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int c = begin + threadIdx.x + i * blockDim.x;
            live[i] = c < end;
            if (live[i]) {
                xv[i] = load_stream(xr + c);
                rv[i] = load_stream(rr + c);
            }
        }
        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            if (!live[i]) continue;
            const uint32_t* xw = reinterpret_cast<const uint32_t*>(&xv[i]);
            const uint32_t* rw = reinterpret_cast<const uint32_t*>(&rv[i]);
            uint32_t* sw = reinterpret_cast<uint32_t*>(&sv[i]);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t packed = pack_bf16x2(bf16_lo(xw[k]) + bf16_lo(rw[k]), bf16_hi(xw[k]) + bf16_hi(rw[k]));
                sw[k] = packed;
                const float s0 = bf16_lo(packed), s1 = bf16_hi(packed);
                ss = fmaf(s0, s0, ss);
                ss = fmaf(s1, s1, ss);
            }
            store_stream(rr + (begin + threadIdx.x + i * blockDim.x), sv[i]);
        }
        ss = cta_allreduce(ss, red_sum, SumOp{});
        ss = cluster_allreduce(ss, &cl_slot[0], ctas_per_row, SumOp{});
        // (reuse of `ss` below: the row's sum of squares)
        const float inv = 1.0f / sqrtf(ss / static_cast<float>(p.hidden) + p.eps);

        uint4 wv[VPT];
#pragma unroll
        for (int i = 0; i < VPT; ++i)
            if (live[i]) wv[i] = load_cached(wr + (begin + threadIdx.x + i * blockDim.x));

        if constexpr (EP == kBf16) {
            uint4* outr = static_cast<uint4*>(p.out) + row * p.nvec;
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                if (!live[i]) continue;
                const uint32_t* sw = reinterpret_cast<const uint32_t*>(&sv[i]);
                const uint32_t* ww = reinterpret_cast<const uint32_t*>(&wv[i]);
                uint4 o;
                uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    ow[k] = pack_bf16x2(bf16_lo(sw[k]) * inv * bf16_lo(ww[k]), bf16_hi(sw[k]) * inv * bf16_hi(ww[k]));
                store_stream(outr + (begin + threadIdx.x + i * blockDim.x), o);
            }
            cluster_sync_if(ctas_per_row);
        } else {
            float qmul;
            if constexpr (EP == kFp8Static) {
                const float sc = __ldg(p.scale);
                qmul = sc > 0.0f ? 1.0f / sc : 0.0f;
            } else {
                float amax = 0.0f;
#pragma unroll
                for (int i = 0; i < VPT; ++i) {
                    if (!live[i]) continue;
                    const uint32_t* sw = reinterpret_cast<const uint32_t*>(&sv[i]);
                    const uint32_t* ww = reinterpret_cast<const uint32_t*>(&wv[i]);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        amax = fmaxf(amax, fabsf(bf16_lo(sw[k]) * inv * bf16_lo(ww[k])));
                        amax = fmaxf(amax, fabsf(bf16_hi(sw[k]) * inv * bf16_hi(ww[k])));
                    }
                }
                amax = cta_allreduce(amax, red_max, MaxOp{});
                amax = cluster_allreduce(amax, &cl_slot[1], ctas_per_row, MaxOp{});
                const float sc = amax / 448.0f;
                qmul = sc > 0.0f ? 1.0f / sc : 0.0f;
                if (rank == 0 && threadIdx.x == 0) p.scale[row] = sc;
            }
            uint2* outr = reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.out) + row * (int64_t)p.nvec * 8);
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                if (!live[i]) continue;
                const uint32_t* sw = reinterpret_cast<const uint32_t*>(&sv[i]);
                const uint32_t* ww = reinterpret_cast<const uint32_t*>(&wv[i]);
                float v[8];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    v[2 * k] = bf16_lo(sw[k]) * inv * bf16_lo(ww[k]) * qmul;
                    v[2 * k + 1] = bf16_hi(sw[k]) * inv * bf16_hi(ww[k]) * qmul;
                }
                uint2 q;
                q.x = pack_e4m3x4(v[0], v[1], v[2], v[3]);
                q.y = pack_e4m3x4(v[4], v[5], v[6], v[7]);
                store_stream(outr + (begin + threadIdx.x + i * blockDim.x), q);
            }
            cluster_sync_if(ctas_per_row);
        }
    }
}

template <int EP>
cudaError_t launch_ep(const NormParams& p, const RowPlan& plan, cudaStream_t s) {
    void (*kern)(NormParams, int, int) = nullptr;
    switch (plan.vpt) {
        case 1: kern = add_rmsnorm_kernel<1, EP>; break;
        case 2: kern = add_rmsnorm_kernel<2, EP>; break;
        case 4: kern = add_rmsnorm_kernel<4, EP>; break;
        case 8: kern = add_rmsnorm_kernel<8, EP>; break;
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
    cfg.numAttrs = plan.ctas_per_row > 1 ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p, plan.ctas_per_row, plan.slice);
}

}  // namespace

cudaError_t launch_add_rmsnorm(const NormParams& p, Epilogue ep, const RowPlan& plan, cudaStream_t s) {
    switch (ep) {
        case kBf16: return launch_ep<kBf16>(p, plan, s);
        case kFp8Static: return launch_ep<kFp8Static>(p, plan, s);
        case kFp8Dynamic: return launch_ep<kFp8Dynamic>(p, plan, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace mbd
