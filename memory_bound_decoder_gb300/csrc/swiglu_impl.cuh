// Per-slice body of the fused SwiGLU over the stacked gate_up row (bf16, FP8 E4M3 or NVFP4 out), shared
// by the one-launch-per-call kernels (swiglu.cu) and the persistent program kernel (program.cu).
#pragma once

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

}  // namespace

struct SwigluSmem {
    PMax part_max[32];
    Exchange ex;
    float row_qmul;
    int ok_flag;
};

// Warm L2 with this thread's gate and up vectors of one row slice.
template <int VPT>
__device__ __forceinline__ void swiglu_prefetch(const SwigluParams p, int64_t row, int begin, int end) {
    const uint4* gr = static_cast<const uint4*>(p.gate_up) + row * (int64_t)p.nvec * 2;
    const uint4* ur = gr + p.nvec;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int c = begin + threadIdx.x + i * blockDim.x;
        if (c < end) {
            prefetch_l2(gr + c);
            prefetch_l2(ur + c);
        }
    }
}

// One CTA's share of one row: vectors [begin, end) of `row` (at most VPT per thread; begin even for
// NVFP4), the CTA being `rank` of the `nctas` CTAs of the row (a cluster when nctas > 1; only the dynamic
// FP8 epilogue reduces over the row). Every thread of the CTA calls it. CL as for norm_row_slice (it
// matters only to the dynamic epilogue).
template <int VPT, int EP, int CL = kRowAny>
__device__ __forceinline__ void swiglu_row_slice(const SwigluParams p, int64_t row, int rank, int nctas, int begin,
                                                 int end, SwigluSmem& sm) {
    PMax* part_max = sm.part_max;
    Exchange& ex = sm.ex;
    const int ctas_per_row = CL == kRowInCta ? 1 : nctas;
    const bool single = CL == kRowInCta || (CL == kRowAny && nctas == 1);
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
    if constexpr (EP == kFp8Dynamic) {
        if (!single) exchange_init(ex, ctas_per_row);   // overlaps the loads in flight
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
            if (single) {   // the whole row in this CTA: one barrier, every thread forms the scale
                const float sc = block_total(PMax{amax}, part_max).v / 448.0f;
                qmul = sc > 0.0f ? 1.0f / sc : 0.0f;
                if (threadIdx.x == 0) p.scale[row] = sc;
            } else {
                if (!row_reduce(PMax{amax}, part_max, ex, rank, ctas_per_row, &sm.ok_flag, [&](PMax t) {
                        const float sc = t.v / 448.0f;
                        sm.row_qmul = sc > 0.0f ? 1.0f / sc : 0.0f;
                        if (rank == 0) p.scale[row] = sc;
                    }))
                    return;
                qmul = sm.row_qmul;
            }
        }
        // formed after the reduction: nothing but the products stays live across the exchange
        uint2* outr = reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.out) + row * (int64_t)p.nvec * 8);
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

// Dynamic FP8 SwiGLU of a whole row wider than one CTA holds (more than VPT vectors per thread), in two
// passes over chunks of blockDim * VPT vectors: max |h| over the row with nothing kept, the row scale, then
// h recomputed from the same gate and up vectors (now in L2; the first pass loads them with the default
// cache policy, the second as a last use) and quantised. The products are computed identically in both
// passes, so the codes equal those of the one-pass form. Every thread of the CTA calls it.
template <int VPT>
__device__ __forceinline__ void swiglu_dynamic_two_pass(const SwigluParams p, int64_t row, SwigluSmem& sm) {
    const uint4* gr = static_cast<const uint4*>(p.gate_up) + row * (int64_t)p.nvec * 2;
    const uint4* ur = gr + p.nvec;
    const int step = blockDim.x * VPT;
    float amax = 0.0f;
    for (int b = 0; b < p.nvec; b += step) {
        uint4 gv[VPT], uv[VPT];
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int c = b + threadIdx.x + i * blockDim.x;
            if (c < p.nvec) {
                gv[i] = load_cached(gr + c);
                uv[i] = load_cached(ur + c);
            }
        }
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            if (b + threadIdx.x + i * blockDim.x >= p.nvec) continue;
            const uint32_t* gw = reinterpret_cast<const uint32_t*>(&gv[i]);
            const uint32_t* uw = reinterpret_cast<const uint32_t*>(&uv[i]);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 h = silu_times(bf16x2_to_float2(gw[k]), bf16x2_to_float2(uw[k]));
                amax = fmaxf(amax, fmaxf(fabsf(h.x), fabsf(h.y)));
            }
        }
    }
    const float sc = block_total(PMax{amax}, sm.part_max).v / 448.0f;
    if (threadIdx.x == 0) p.scale[row] = sc;
    const float2 q2 = f2(sc > 0.0f ? 1.0f / sc : 0.0f);
    uint2* outr = reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.out) + row * (int64_t)p.nvec * 8);
    for (int b = 0; b < p.nvec; b += step) {
        uint4 gv[VPT], uv[VPT];
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int c = b + threadIdx.x + i * blockDim.x;
            if (c < p.nvec) {
                gv[i] = load_stream(gr + c);
                uv[i] = load_stream(ur + c);
            }
        }
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int c = b + threadIdx.x + i * blockDim.x;
            if (c >= p.nvec) continue;
            const uint32_t* gw = reinterpret_cast<const uint32_t*>(&gv[i]);
            const uint32_t* uw = reinterpret_cast<const uint32_t*>(&uv[i]);
            float2 h[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) h[k] = silu_times(bf16x2_to_float2(gw[k]), bf16x2_to_float2(uw[k]));
            uint2 q;
            q.x = pack_e4m3x4(__fmul2_rn(h[0], q2), __fmul2_rn(h[1], q2));
            q.y = pack_e4m3x4(__fmul2_rn(h[2], q2), __fmul2_rn(h[3], q2));
            store_stream(outr + c, q);
        }
    }
}

}  // namespace mbd
