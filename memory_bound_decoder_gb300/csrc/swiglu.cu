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
#include "common.cuh"
#include "launch.h"

namespace mbd {

namespace {

// silu(g) * u = g * u / (1 + e^-g) for a pair of elements, with packed fp32x2 arithmetic (FFMA2/FMUL2/
// FADD2) around the two hardware transcendentals. e^-g = 2^(-g log2 e) comes from the base-2 exponential
// (ex2.approx) of the fp32-rounded argument t, times 2^d ~ 1 + d ln 2 for the rounding residual
// d = -g log2 e - t (exact through an FMA plus the low part of log2 e), so the error does not grow with |g|;
// 1 / (1 + e) comes from the hardware reciprocal (rcp.approx). For g below about -88, e overflows to +inf
// (the correction factor is positive, so no NaN), 1 / (1 + e) is 0 and the result is a signed zero, where
// the exact value is below 1e-36 in magnitude.
__device__ __forceinline__ float ex2_approx(float t) {
    float e;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(t));
    return e;
}

__device__ __forceinline__ float2 silu_times(float2 g, float2 u) {
    constexpr float kLog2e = 1.44269502162933349609375f;   // log2(e) rounded to fp32
    constexpr float kLog2eLo = 1.925963033500011e-08f;     // log2(e) - kLog2e
    constexpr float kLn2 = 0.693147182464599609375f;
    const float2 t = __fmul2_rn(g, f2(-kLog2e));
    const float2 d = __ffma2_rn(g, f2(-kLog2eLo), __ffma2_rn(g, f2(-kLog2e), make_float2(-t.x, -t.y)));
    float2 e = make_float2(ex2_approx(t.x), ex2_approx(t.y));
    e = __fmul2_rn(e, __ffma2_rn(d, f2(kLn2), f2(1.0f)));
    const float2 den = __fadd2_rn(e, f2(1.0f));
    const float2 r = make_float2(rcp_approx_ftz(den.x), rcp_approx_ftz(den.y));
    return __fmul2_rn(__fmul2_rn(g, r), u);
}

template <int VPT, int EP>
__global__ void __launch_bounds__(512, VPT <= 2 ? 4 : 1) swiglu_kernel(SwigluParams p, int ctas_per_row, int slice, int prefetch) {
    __shared__ PMax part_max[32];
    __shared__ Exchange ex;
    __shared__ float row_qmul;
    __shared__ int ok_flag;

    const int64_t row = launch_row();
    if (row >= p.rows) return;   // past the last row (the whole cluster shares the row)
    const int rank = static_cast<int>(blockIdx.x);
    const int begin = rank * slice;
    const int end = min(begin + slice, p.nvec);

    const uint4* gr = static_cast<const uint4*>(p.gate_up) + row * (int64_t)p.nvec * 2;
    const uint4* ur = gr + p.nvec;

    pdl_trigger();
    if (prefetch) {
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int c = begin + threadIdx.x + i * blockDim.x;
        if (c < end) {
            prefetch_l2(gr + c);
            prefetch_l2(ur + c);
        }
    }
    }
    pdl_wait();

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
    if constexpr (EP == kFp8Dynamic) {
        if (ctas_per_row > 1) exchange_init(ex, ctas_per_row);   // overlaps the loads in flight
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
            for (int k = 0; k < 4; ++k) ow[k] = pack_bf16x2(silu_times(bf16x2_to_float2(gw[k]), bf16x2_to_float2(uw[k])));
            store_stream(outr + (begin + threadIdx.x + i * blockDim.x), o);
        }
    } else if constexpr (EP == kNvfp4) {
        // NVFP4 from registers, one vector at a time: the block maximum of 16 elements comes from this lane
        // and its neighbour (slices start on an even vector).
        const Nvfp4Row nr = nvfp4_unit_row(nvfp4_tensor_scale(p.scale));
        unsigned int* qr = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(p.out) + row * (int64_t)p.nvec * 4);
        uint8_t* sfr = p.out_sf + row * (int64_t)(p.nvec / 2);
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            float2 h[4];
            const uint32_t* gw = reinterpret_cast<const uint32_t*>(&gv[i]);
            const uint32_t* uw = reinterpret_cast<const uint32_t*>(&uv[i]);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                h[k] = live[i] ? silu_times(bf16x2_to_float2(gw[k]), bf16x2_to_float2(uw[k])) : f2(0.0f);
            uint32_t sf;
            const uint32_t q = nvfp4_encode(h, nr, &sf);   // whole warp (block max by shuffle)
            if (!live[i]) continue;
            const int c = begin + threadIdx.x + i * blockDim.x;
            store_stream(qr + c, q);
            if ((threadIdx.x & 1) == 0) sfr[c >> 1] = static_cast<uint8_t>(sf);
        }
    } else {
        uint2* outr = reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.out) + row * (int64_t)p.nvec * 8);
        float2 h[VPT][4];
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
                h[i][k] = silu_times(bf16x2_to_float2(gw[k]), bf16x2_to_float2(uw[k]));
                if constexpr (EP == kFp8Dynamic) amax = fmaxf(amax, fmaxf(fabsf(h[i][k].x), fabsf(h[i][k].y)));
            }
        }
        if constexpr (EP == kFp8Dynamic) {
            if (!row_reduce(PMax{amax}, part_max, ex, rank, ctas_per_row, &ok_flag, [&](PMax t) {
                    const float sc = t.v / 448.0f;
                    row_qmul = sc > 0.0f ? 1.0f / sc : 0.0f;
                    if (rank == 0) p.scale[row] = sc;
                }))
                return;
            qmul = row_qmul;
        }
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            if (!live[i]) continue;
            const float2 q2 = f2(qmul);
            uint2 q;
            q.x = pack_e4m3x4(__fmul2_rn(h[i][0], q2), __fmul2_rn(h[i][1], q2));
            q.y = pack_e4m3x4(__fmul2_rn(h[i][2], q2), __fmul2_rn(h[i][3], q2));
            store_stream(outr + (begin + threadIdx.x + i * blockDim.x), q);
        }
    }
}

template <int EP>
cudaError_t launch_ep(const SwigluParams& p, const RowPlan& plan, cudaStream_t s) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    const int cluster = EP == kFp8Dynamic ? plan.ctas_per_row : 1;
    void (*kern)(SwigluParams, int, int, int) = nullptr;
    switch (plan.vpt) {
        case 1: kern = swiglu_kernel<1, EP>; break;
        case 2: kern = swiglu_kernel<2, EP>; break;
        case 4: kern = swiglu_kernel<4, EP>; break;
        case 8: kern = swiglu_kernel<8, EP>; break;
        default: return cudaErrorInvalidValue;
    }
    fill_launch(cfg, attr, p.rows, plan.ctas_per_row, plan.threads, cluster, s);
    return cudaLaunchKernelEx(&cfg, kern, p, plan.ctas_per_row, plan.slice, plan.prefetch);
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
