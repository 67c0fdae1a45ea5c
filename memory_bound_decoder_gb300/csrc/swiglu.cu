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
// from the registers, so the activation crosses HBM exactly once. For large batches of wide rows its inputs
// arrive by two bulk copies per CTA into shared memory instead (swiglu_dyn_bulk_kernel), which leaves the
// registers to the products and lets more CTAs, and more bytes in flight, share an SM.
#include <atomic>

#include "swiglu_impl.cuh"

namespace mbd {

namespace {

template <int VPT, int EP, int CL>
__global__ void __launch_bounds__(512, VPT <= 2 ? 4 : 1) swiglu_kernel(const __grid_constant__ SwigluParams p, int ctas_per_row, int slice, int prefetch,
                                                                   int ahead, int order) {
    __shared__ SwigluSmem sm;
    const int64_t row = launch_row();
    if (row >= p.rows) return;   // past the last row (the whole cluster shares the row)
    const int rank = static_cast<int>(blockIdx.x);
    const int begin = rank * slice;
    const int end = min(begin + slice, p.nvec);
    pdl_enter_trigger(order);
    if (prefetch) swiglu_prefetch<VPT>(p, row, begin, end);
    pdl_enter_wait(order);
    // The row a later wave will run here is fetched into L2 now, so that its loads meet L2 instead of HBM;
    // the bytes come from HBM once either way (the rows in flight plus those ahead fit L2 many times over).
    // Two bulk prefetches (gate and up slices) from one thread.
    if (ahead > 0 && row + ahead < p.rows && threadIdx.x == 0) {
        const uint4* gr = static_cast<const uint4*>(p.gate_up) + (row + ahead) * (int64_t)p.nvec * 2 + begin;
        const uint32_t bytes = static_cast<uint32_t>(end - begin) * 16u;
        prefetch_l2_bulk(gr, bytes);
        prefetch_l2_bulk(gr + p.nvec, bytes);
    }
    swiglu_row_slice<VPT, EP, CL>(p, row, rank, ctas_per_row, begin, end, sm);
    pdl_leave(order);
}

// Dynamic FP8 SwiGLU with the CTA's gate and up slices brought into shared memory by two bulk copies
// (cp.async.bulk, completion counted on an mbarrier) instead of per-thread loads into registers: registers
// then hold only the fp32 products, so more CTAs (and more bytes in flight) fit on an SM while others sit in
// their row reduction. Same arithmetic, reduction and stores as swiglu_row_slice. Rows always span a cluster
// (ctas_per_row >= 2; the planner uses 7 or 8).
struct BulkSmem {
    unsigned long long load_bar;
};

template <int VPT>
__device__ __forceinline__ void swiglu_dyn_bulk_row(const SwigluParams& p, int64_t row, int ctas_per_row, int slice,
                                                    int ahead, int order, uint4* slices, SwigluSmem& sm,
                                                    BulkSmem& bs) {
    const int rank = static_cast<int>(blockIdx.x);
    const int begin = rank * slice;
    const int end = min(begin + slice, p.nvec);
    const int n = end - begin;
    const uint32_t bar = smem_addr(&bs.load_bar);
    pdl_enter_trigger(order);
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    pdl_enter_wait(order);
    if (threadIdx.x == 0) {
        const uint4* gr = static_cast<const uint4*>(p.gate_up) + row * (int64_t)p.nvec * 2 + begin;
        const uint32_t bytes = static_cast<uint32_t>(n) * 16u;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(2u * bytes) : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     ::"r"(smem_addr(slices)), "l"(gr), "r"(bytes), "r"(bar) : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     ::"r"(smem_addr(slices + slice)), "l"(gr + p.nvec), "r"(bytes), "r"(bar) : "memory");
        if (ahead > 0 && row + ahead < p.rows) {   // warm L2 with the row a later wave runs here
            prefetch_l2_bulk(gr + ahead * (int64_t)p.nvec * 2, bytes);
            prefetch_l2_bulk(gr + ahead * (int64_t)p.nvec * 2 + p.nvec, bytes);
        }
    }
    exchange_init(sm.ex, ctas_per_row);   // its cluster barrier overlaps the copies
    // every thread waits for both slices (bounded; on expiry: error flag, and the copies are waited for once
    // more before the CTA may leave, since they write into its shared memory)
    bool landed = false;
    {
        const long long t0 = clock64();
        uint32_t done = 0;
        while (true) {
            asm volatile("{\n .reg .pred q;\n mbarrier.try_wait.parity.shared::cta.b64 q, [%1], 0;\n selp.u32 %0, 1, 0, q;\n}"
                         : "=r"(done) : "r"(bar) : "memory");
            if (done || clock64() - t0 > kWaitLimitCycles) break;
        }
        landed = done != 0;
        if (!landed) {
            if (threadIdx.x == 0) atomicOr(&g_device_error_flags, kDevErrExchangeTimeout);
            const long long t1 = clock64();
            while (!done && clock64() - t1 < kWaitLimitCycles)
                asm volatile("{\n .reg .pred q;\n mbarrier.try_wait.parity.shared::cta.b64 q, [%1], 0;\n selp.u32 %0, 1, 0, q;\n}"
                             : "=r"(done) : "r"(bar) : "memory");
        }
    }
    float2 h[VPT][4];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int c = threadIdx.x + i * blockDim.x;
        if (c >= n || !landed) continue;
        const uint4 gv = slices[c], uv = slices[slice + c];
        const uint32_t* gw = reinterpret_cast<const uint32_t*>(&gv);
        const uint32_t* uw = reinterpret_cast<const uint32_t*>(&uv);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            h[i][k] = silu_times(bf16x2_to_float2(gw[k]), bf16x2_to_float2(uw[k]));
            amax = fmaxf(amax, fmaxf(fabsf(h[i][k].x), fabsf(h[i][k].y)));
        }
    }
    if (!row_reduce(PMax{amax}, sm.part_max, sm.ex, rank, ctas_per_row, &sm.ok_flag, [&](PMax t) {
            const float sc = t.v / 448.0f;
            sm.row_qmul = sc > 0.0f ? 1.0f / sc : 0.0f;
            if (rank == 0) p.scale[row] = sc;
        }))
        return;
    const float qmul = sm.row_qmul;
    if (!landed) return;
    uint2* outr = reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.out) + row * (int64_t)p.nvec * 8) + begin;
    const float2 q2 = f2(qmul);
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int c = threadIdx.x + i * blockDim.x;
        if (c >= n) continue;
        uint2 q;
        q.x = pack_e4m3x4(__fmul2_rn(h[i][0], q2), __fmul2_rn(h[i][1], q2));
        q.y = pack_e4m3x4(__fmul2_rn(h[i][2], q2), __fmul2_rn(h[i][3], q2));
        store_stream(outr + c, q);
    }
}

template <int VPT>
__global__ void __launch_bounds__(320, 4) swiglu_dyn_bulk_kernel(const __grid_constant__ SwigluParams p, int ctas_per_row,
                                                                 int slice, int ahead, int order) {
    extern __shared__ __align__(16) uint4 slices[];   // gate slice [0, slice), up slice [slice, 2 slice)
    __shared__ SwigluSmem sm;
    __shared__ BulkSmem bs;
    const int64_t row = launch_row();
    if (row >= p.rows) return;   // past the last row (the whole cluster shares the row)
    swiglu_dyn_bulk_row<VPT>(p, row, ctas_per_row, slice, ahead, order, slices, sm, bs);
    pdl_leave(order);
}

// Per device (up to 64): the id of the context in which the bulk kernel's preferred carveout, the largest
// shared-memory share, was last requested, so that the SM's shared memory rather than its L1 share bounds
// the resident CTAs (each holds two row slices, up to 40 KB). A kernel attribute belongs to a context: a
// context re-created on the device (cudaDeviceReset) gets the request again; with no context id (0) every
// launch requests it.
std::atomic<unsigned long long> g_bulk_carveout_ctx[kMaxCachedDevices];

cudaError_t launch_dyn_bulk(const SwigluParams& p, const RowPlan& plan, cudaStream_t s) {
    if (plan.vpt != 4 || plan.ctas_per_row < 2 || plan.ctas_per_row > kMaxClusterCtas) return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long ctx = current_context_id();
    if (dev < 0 || dev >= kMaxCachedDevices || ctx == 0 ||
        g_bulk_carveout_ctx[dev].load(std::memory_order_acquire) != ctx) {
        e = cudaFuncSetAttribute(swiglu_dyn_bulk_kernel<4>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 static_cast<int>(cudaSharedmemCarveoutMaxShared));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kMaxCachedDevices) g_bulk_carveout_ctx[dev].store(ctx, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    fill_launch(cfg, attr, p.rows, plan.ctas_per_row, plan.threads, plan.ctas_per_row, s);
    cfg.dynamicSmemBytes = static_cast<size_t>(plan.slice) * 32;
    return cudaLaunchKernelEx(&cfg, swiglu_dyn_bulk_kernel<4>, p, plan.ctas_per_row, plan.slice, plan.ahead, plan.order);
}

template <int EP>
cudaError_t launch_ep(const SwigluParams& p, const RowPlan& plan, cudaStream_t s) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    const int cluster = EP == kFp8Dynamic ? plan.ctas_per_row : 1;
    void (*kern)(SwigluParams, int, int, int, int, int) = nullptr;
    // only the dynamic epilogue reduces over the row; the streams compile no reduction either way
    constexpr int kMulti = EP == kFp8Dynamic ? kRowInCluster : kRowInCta;
    const bool cl = cluster > 1;
    switch (plan.vpt) {
        case 1: kern = cl ? swiglu_kernel<1, EP, kMulti> : swiglu_kernel<1, EP, kRowInCta>; break;
        case 2: kern = cl ? swiglu_kernel<2, EP, kMulti> : swiglu_kernel<2, EP, kRowInCta>; break;
        case 4: kern = cl ? swiglu_kernel<4, EP, kMulti> : swiglu_kernel<4, EP, kRowInCta>; break;
        case 8: kern = cl ? swiglu_kernel<8, EP, kMulti> : swiglu_kernel<8, EP, kRowInCta>; break;
        default: return cudaErrorInvalidValue;
    }
    if (EP == kFp8Dynamic && plan.bulk) return launch_dyn_bulk(p, plan, s);
    fill_launch(cfg, attr, p.rows, plan.ctas_per_row, plan.threads, cluster, s);
    return cudaLaunchKernelEx(&cfg, kern, p, plan.ctas_per_row, plan.slice, plan.prefetch, plan.ahead, plan.order);
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
