// Device-side building blocks shared by the fused kernels: 16-byte vector loads and stores with
// streaming cache hints, bf16 and E4M3 packing, and the per-row reduction (warp shuffles, a shared-memory
// step across warps, and a distributed-shared-memory step across the CTAs of a thread-block cluster).
#pragma once

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mbd {

namespace cg = cooperative_groups;

// ------------------------------------------------------------------------------------------ memory

// Streaming loads/stores: every activation byte is touched exactly once, so ask the caches to evict
// it first (ld/st .cs). The weight is re-read by every row and uses the default (cached) path.
__device__ __forceinline__ uint4 load_stream(const uint4* p) { return __ldcs(p); }
__device__ __forceinline__ void store_stream(uint4* p, const uint4& v) { __stcs(p, v); }
__device__ __forceinline__ void store_stream(uint2* p, const uint2& v) { __stcs(p, v); }
__device__ __forceinline__ uint4 load_cached(const uint4* p) { return __ldg(p); }

// ------------------------------------------------------------------------------------------ bf16 / e4m3

// A 32-bit word holds two bf16 values: element 2k in the low half, element 2k+1 in the high half.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Round two fp32 values to bf16 (nearest even) and pack them (lo -> low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&p);
}

// Round two fp32 values to E4M3 (nearest even, finite overflow saturates to +-448) and pack them:
// lo lands in the low byte, i.e. at the lower address once stored.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
    return pack_e4m3x2(a, b) | (pack_e4m3x2(c, d) << 16);
}

// ------------------------------------------------------------------------------------------ reductions

struct SumOp {
    __device__ __forceinline__ float operator()(float a, float b) const { return a + b; }
};
struct MaxOp {
    __device__ __forceinline__ float operator()(float a, float b) const { return fmaxf(a, b); }
};

// Butterfly (xor) reduction: every lane ends with the same value because each step combines the same
// two operands on both partner lanes.
template <class Op>
__device__ __forceinline__ float warp_allreduce(float v, Op op) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// CTA-wide reduction; every thread returns the same total. Inputs are sums or magnitudes (>= 0), so 0
// is the identity for both operators. `scratch` holds one float per warp and may be
// reused only after a __syncthreads() that follows this call.
template <class Op>
__device__ __forceinline__ float cta_allreduce(float v, float* scratch, Op op) {
    v = warp_allreduce(v, op);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    const int nwarps = (blockDim.x + 31) >> 5;
    float t = lane < nwarps ? scratch[lane] : 0.0f;
    return warp_allreduce(t, op);
}

// Combine the CTA totals of the `nctas` CTAs of this cluster (they all compute the same value, summed in
// rank order). `slot` is a __shared__ float of this CTA. The caller must cluster-sync again before `slot`
// is rewritten or before the CTA exits, because other CTAs read it remotely.
template <class Op>
__device__ __forceinline__ float cluster_allreduce(float cta_total, float* slot, int nctas, Op op) {
    if (nctas == 1) return cta_total;
    cg::cluster_group cluster = cg::this_cluster();
    if (threadIdx.x == 0) *slot = cta_total;
    cluster.sync();
    const int lane = threadIdx.x & 31;
    float t = 0.0f;
    if (lane < nctas) t = *cluster.map_shared_rank(slot, lane);
    return warp_allreduce(t, op);
}

__device__ __forceinline__ void cluster_sync_if(int nctas) {
    if (nctas > 1) cg::this_cluster().sync();
}

}  // namespace mbd
