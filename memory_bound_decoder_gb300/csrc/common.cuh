// Device-side building blocks shared by the fused kernels: 16-byte vector loads and stores with
// streaming cache hints, bf16 and E4M3 packing, and the per-row reduction (warp shuffles, a shared-memory
// step across warps, and a distributed-shared-memory step across the CTAs of a thread-block cluster).
#pragma once

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "launch.h"

namespace mbd {

namespace cg = cooperative_groups;

// ------------------------------------------------------------------------------------------ memory

// Streaming loads/stores: every activation byte is touched exactly once, so ask the caches to evict
// it first (ld/st .cs). The weight is re-read by every row and uses the default (cached) path.
__device__ __forceinline__ uint4 load_stream(const uint4* p) { return __ldcs(p); }
__device__ __forceinline__ void store_stream(uint4* p, const uint4& v) { __stcs(p, v); }
__device__ __forceinline__ void store_stream(uint2* p, const uint2& v) { __stcs(p, v); }
__device__ __forceinline__ void store_stream(unsigned int* p, unsigned int v) { __stcs(p, v); }
__device__ __forceinline__ uint4 load_cached(const uint4* p) { return __ldg(p); }

// ------------------------------------------------------------------------------------------ bf16 / e4m3

// Lane-wise bf16 maximum and minimum of two pairs given as bits (for non-negative values: magnitudes).
__device__ __forceinline__ uint32_t max_bf16x2_bits(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t min_bf16x2_bits(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// A 32-bit word holds two bf16 values: element 2k in the low half, element 2k+1 in the high half.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Both halves of a bf16x2 word as a float2 (exact).
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }

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

__device__ __forceinline__ uint32_t pack_bf16x2(float2 v) { return pack_bf16x2(v.x, v.y); }
__device__ __forceinline__ uint32_t pack_e4m3x4(float2 a, float2 b) { return pack_e4m3x4(a.x, a.y, b.x, b.y); }

// ------------------------------------------------------------------------------------------ NVFP4

// Eight fp32 values to E2M1 (nearest even, saturating to +-6), packed into one word: element 0 in the
// lowest nibble, so element 2i lands in the low nibble of byte i once stored.
__device__ __forceinline__ uint32_t pack_e2m1x8(float2 a, float2 b, float2 c, float2 d) {
    uint32_t r;
    asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
        "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
        : "=r"(r)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y), "f"(d.x), "f"(d.y));
    return r;
}

// Value of an E4M3 code (low byte of `code`) through the hardware conversion E4M3 -> f16 -> f32 (exact).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<unsigned short>(code & 0xffu)));
    float f;
    asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(static_cast<unsigned short>(h2 & 0xffffu)));
    return f;
}

__device__ __forceinline__ float rcp_approx_ftz(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// The per-tensor fp32 scale S of an NVFP4 output, read once per thread. S outside [2^-64, 2^64] (or not a
// number) counts as unusable and gives zero block scales and zero codes everywhere.
__device__ __forceinline__ float nvfp4_tensor_scale_of(float s) { return (s >= 0x1p-64f && s <= 0x1p64f) ? s : 0.0f; }
__device__ __forceinline__ float nvfp4_tensor_scale(const float* scale) { return nvfp4_tensor_scale_of(__ldg(scale)); }

// Row constants of the NVFP4 epilogue for row values v = y * vmul under the tensor scale S (0 when
// unusable): k = vmul / (6 S) turns a block maximum of |y| into the block scale's argument, and
// ms = vmul / S turns y into v / S. Two IEEE divisions per thread, none per element.
struct Nvfp4Row {
    float k;
    float ms;
};

__device__ __forceinline__ Nvfp4Row nvfp4_row(float vmul, float s) {
    if (s == 0.0f) return Nvfp4Row{0.0f, 0.0f};
    return Nvfp4Row{vmul / (6.0f * s), vmul / s};
}

// The same for vmul == 1 through correctly rounded reciprocals (equal to 1 / x, cheaper than a division).
__device__ __forceinline__ Nvfp4Row nvfp4_unit_row(float s) {
    if (s == 0.0f) return Nvfp4Row{0.0f, 0.0f};
    return Nvfp4Row{__frcp_rn(6.0f * s), __frcp_rn(s)};
}

// NVFP4 epilogue of one 16-byte vector: eight values y that form half of a 16-element block whose other
// half sits in the neighbouring lane (lane ^ 1). Every lane of the warp must call it (the block maximum is
// shared through a shuffle); a lane without a vector passes zeros. With v = y * vmul:
//     sf   = E4M3(max |v| / (6 S))            = cvt(max |y| * k)
//     code = E2M1(v / (dec(sf) S))            = cvt(y * (ms * (1 / dec(sf))))
// and zero codes when sf is zero. 1 / dec(sf) comes from rcp.approx (within an ulp); with the products the
// code arguments sit within a few ulps of the exact ratios. Returns the packed codes; *sf gets the scale.
__device__ __forceinline__ uint32_t nvfp4_encode(const float2 (&y)[4], const Nvfp4Row& r, uint32_t* sf) {
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k) amax = fmaxf(amax, fmaxf(fabsf(y[k].x), fabsf(y[k].y)));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    const uint32_t code = pack_e4m3x2(amax * r.k, 0.0f) & 0xffu;
    *sf = code;
    const float2 m = f2(r.ms * rcp_approx_ftz(e4m3_value(code)));
    const uint32_t q = pack_e2m1x8(__fmul2_rn(y[0], m), __fmul2_rn(y[1], m), __fmul2_rn(y[2], m), __fmul2_rn(y[3], m));
    return code != 0u ? q : 0u;
}

// ------------------------------------------------------------------------------------------ cluster exchange

// Device-side error word of each kernel translation unit (internal linkage, one per .cu file), read on
// the host through mbd_device_error_flags(). Bits: kDevErrExchangeTimeout.
static __device__ unsigned int g_device_error_flags;
constexpr unsigned int kDevErrExchangeTimeout = 1u;
// Bound of every spin-wait, in SM clock cycles (about one second at 2 GHz).
constexpr long long kWaitLimitCycles = 2LL << 30;

// Partial results of the CTAs of one row are exchanged through distributed shared memory: every CTA
// pushes its 16-byte partial into slot[my_rank] of every peer with st.async, whose completion is counted
// on the peer's mbarrier (transaction bytes). No cluster-wide release fence is needed, so the exchange
// does not wait for this CTA's outstanding global stores. A CTA leaves only after its own mbarrier has
// seen every peer's bytes, so no write can target a CTA that has exited.
constexpr int kMaxClusterCtas = 8;   // portable cluster size

// Where a row reduction runs, as a compile-time choice of the row-slice bodies: the row in one CTA, the row
// over a cluster, or either (decided by the CTA count at run time).
constexpr int kRowAny = 0, kRowInCta = 1, kRowInCluster = 2;

struct alignas(16) Exchange {
    float4 slot[kMaxClusterCtas];
    unsigned long long mbar;
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Call once per CTA, by all threads, before any peer may push (it ends with a cluster barrier).
__device__ __forceinline__ void exchange_init(Exchange& ex, int nctas) {
    if (threadIdx.x == 0) {
        const uint32_t mb = smem_addr(&ex.mbar);
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mb) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb), "r"((nctas - 1) * 16)
                     : "memory");
    }
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Called by warp 0 only: lane 0 publishes this CTA's partial in its own slot, lanes 0..nctas-1 push it
// into the same slot of every peer.
__device__ __forceinline__ void exchange_send(Exchange& ex, float4 v, int my_rank, int nctas) {
    const int lane = threadIdx.x & 31;
    if (lane == 0) ex.slot[my_rank] = v;
    if (lane < nctas && lane != my_rank) {
        uint32_t rslot, rbar;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rslot) : "r"(smem_addr(&ex.slot[my_rank])), "r"(lane));
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rbar) : "r"(smem_addr(&ex.mbar)), "r"(lane));
        asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
                     ::"r"(rslot), "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)), "r"(__float_as_uint(v.z)),
                       "r"(__float_as_uint(v.w)), "r"(rbar)
                     : "memory");
    }
}

// Called by warp 0 only: lane 0 polls the mbarrier until every peer's bytes have landed (phase 0), then
// the warp synchronises so that all its lanes may read slot[]. Gives up after kWaitLimitCycles, sets
// kDevErrExchangeTimeout and returns false on every lane.
__device__ __forceinline__ bool exchange_wait_warp(Exchange& ex, long long limit = kWaitLimitCycles) {
    uint32_t done = 0;
    if ((threadIdx.x & 31) == 0) {
        const uint32_t mb = smem_addr(&ex.mbar);
        const long long t0 = clock64();
        while (true) {
            asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n selp.u32 %0, 1, 0, p;\n}"
                         : "=r"(done)
                         : "r"(mb)
                         : "memory");
            if (done || clock64() - t0 > limit) break;
        }
        if (!done) atomicOr(&g_device_error_flags, kDevErrExchangeTimeout);
    }
    __syncwarp();
    return __shfl_sync(0xffffffffu, done, 0) != 0;
}

// ------------------------------------------------------------------------------------------ row reduction

// Partial results reduced over a row. Each provides combine (commutative in its exact result, so a
// butterfly leaves every lane identical), shuffles, and packing into the 16-byte exchange slot.
struct PSum {
    float v;
    __device__ __forceinline__ static PSum combine(PSum a, PSum b) { return PSum{a.v + b.v}; }
    __device__ __forceinline__ PSum shfl_xor(int o) const { return PSum{__shfl_xor_sync(0xffffffffu, v, o)}; }
    __device__ __forceinline__ float4 pack() const { return make_float4(v, 0.0f, 0.0f, 0.0f); }
    __device__ __forceinline__ static PSum unpack(float4 f) { return PSum{f.x}; }
    __device__ __forceinline__ static PSum zero() { return PSum{0.0f}; }
};

struct PMax {   // of magnitudes (>= 0)
    float v;
    __device__ __forceinline__ static PMax combine(PMax a, PMax b) { return PMax{fmaxf(a.v, b.v)}; }
    __device__ __forceinline__ PMax shfl_xor(int o) const { return PMax{__shfl_xor_sync(0xffffffffu, v, o)}; }
    __device__ __forceinline__ float4 pack() const { return make_float4(v, 0.0f, 0.0f, 0.0f); }
    __device__ __forceinline__ static PMax unpack(float4 f) { return PMax{f.x}; }
    __device__ __forceinline__ static PMax zero() { return PMax{0.0f}; }
};

template <class P>
__device__ __forceinline__ P warp_allreduce_p(P v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = P::combine(v, v.shfl_xor(o));
    return v;
}

// Reduce one value per thread over the whole row. Every warp reduces its lanes; warp 0 combines the warps
// and, when the row spans a cluster, pushes the CTA's partial to the peers and combines theirs in rank
// order (the same order in every CTA, so all CTAs of the row get identical bits); then `fin` runs on warp 0
// lane 0 with the row total and may publish derived constants to shared memory before the closing barrier.
// The other warps issue nothing while they wait at the two CTA barriers. Returns false (in every thread)
// if the cluster exchange timed out.
template <class P, class Fin>
__device__ __forceinline__ bool row_reduce(P mine, P* warp_part, Exchange& ex, int rank, int nctas, int* ok_flag,
                                           Fin fin) {
    mine = warp_allreduce_p(mine);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) warp_part[warp] = mine;
    __syncthreads();
    if (warp == 0) {
        const int nwarps = (blockDim.x + 31) >> 5;
        P t = warp_allreduce_p(lane < nwarps ? warp_part[lane] : P::zero());
        bool ok = true;
        if (nctas > 1) {
            exchange_send(ex, t.pack(), rank, nctas);
            ok = exchange_wait_warp(ex);
            t = P::unpack(ex.slot[0]);
            for (int r = 1; r < nctas; ++r) t = P::combine(t, P::unpack(ex.slot[r]));
        }
        if (lane == 0) {
            *ok_flag = ok;
            if (ok) fin(t);
        }
    }
    __syncthreads();
    return *ok_flag != 0;
}

// Total over a row held by ONE CTA, returned to every thread: the warps reduce their lanes, then every
// thread combines the warp partials in warp order (the same order everywhere, so all threads get identical
// bits). One CTA barrier. warp_part must not be written again before the CTA has passed another barrier
// (the callers' next barrier, or the end of the CTA).
template <class P>
__device__ __forceinline__ P block_total(P mine, P* warp_part) {
    mine = warp_allreduce_p(mine);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) warp_part[warp] = mine;
    __syncthreads();
    const int nwarps = (blockDim.x + 31) >> 5;
    P t = warp_part[0];
    for (int w = 1; w < nwarps; ++w) t = P::combine(t, warp_part[w]);
    return t;
}

// Four warp partials read as one 16-byte vector, slots from `first` on past the last warp counting as zero,
// combined as a pairwise tree.
template <class P>
__device__ __forceinline__ P combine4(float4 f, int first, int nwarps) {
    const P a = first < nwarps ? P{f.x} : P::zero(), b = first + 1 < nwarps ? P{f.y} : P::zero();
    const P c = first + 2 < nwarps ? P{f.z} : P::zero(), d = first + 3 < nwarps ? P{f.w} : P::zero();
    return P::combine(P::combine(a, b), P::combine(c, d));
}

// block_total for a chain of reductions on the critical path (the decode programs' chained norms): every
// thread reads all warp partials at once (16 bytes at a time) and combines them in a fixed pairwise tree
// (the same order everywhere, so all threads get identical bits) instead of a chain of dependent
// shared-memory loads and adds. warp_part: one float per partial, 32 slots, 16-byte aligned. (Compiled into
// the single-call kernels, even in a branch they do not take, it cost them about 1% in their other paths, so
// they keep block_total.)
template <class P>
__device__ __forceinline__ P block_total_tree(P mine, P* warp_part) {
    static_assert(sizeof(P) == sizeof(float), "one-float partials");
    mine = warp_allreduce_p(mine);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) warp_part[warp] = mine;
    __syncthreads();
    const int nwarps = (blockDim.x + 31) >> 5;
    const float4* q = reinterpret_cast<const float4*>(warp_part);
    if (nwarps <= 4) return combine4<P>(q[0], 0, nwarps);
    if (nwarps <= 8) return P::combine(combine4<P>(q[0], 0, nwarps), combine4<P>(q[1], 4, nwarps));
    const P lo = P::combine(P::combine(combine4<P>(q[0], 0, nwarps), combine4<P>(q[1], 4, nwarps)),
                            P::combine(combine4<P>(q[2], 8, nwarps), combine4<P>(q[3], 12, nwarps)));
    if (nwarps <= 16) return lo;
    const P hi = P::combine(P::combine(combine4<P>(q[4], 16, nwarps), combine4<P>(q[5], 20, nwarps)),
                            P::combine(combine4<P>(q[6], 24, nwarps), combine4<P>(q[7], 28, nwarps)));
    return P::combine(lo, hi);
}

// ------------------------------------------------------------------------------------------ PDL

// Programmatic dependent launch: pdl_trigger lets the next kernel in the stream be scheduled as soon as
// every CTA of this one has started; pdl_wait blocks until the previous kernel has completed and its memory
// is visible, and must precede every global load or store. Both are no-ops when the launch did not enable
// programmatic stream serialization.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// The single-call kernels order themselves against the previous kernel by RowPlan::order (PdlOrder, launch.h):
// pdl_enter_trigger first, pdl_enter_wait before the first global load or store (what comes between may only
// warm L2), pdl_leave after the last store.
//   kPdlWaitFirst: trigger, wait                 (every single call)
//   kPdlHead:      wait, trigger                 (first launch of a batch of independent ops: no later launch
//                                                 of the batch starts before the work ahead of it is done)
//   kPdlOverlap:   trigger, ..., wait at exit    (later launches of the batch: they run beside the previous
//                                                 launch, and none completes before its predecessor, so the
//                                                 batch still completes in stream order)
__device__ __forceinline__ void pdl_enter_trigger(int order) {
    if (order != kPdlHead) pdl_trigger();
}
__device__ __forceinline__ void pdl_enter_wait(int order) {
    if (order != kPdlOverlap) pdl_wait();
    if (order == kPdlHead) pdl_trigger();
}
__device__ __forceinline__ void pdl_leave(int order) {
    if (order == kPdlOverlap) pdl_wait();
}

// Warm L2 with a 16-byte vector this thread will load after pdl_wait. A prefetch returns no data, and L2 is
// the point of coherence for global memory, so the load that follows the wait still observes every write
// of the previous kernel; issuing it early only overlaps the HBM latency with the previous kernel's tail.
// Used for small (single-wave, latency-bound) launches only: in a multi-wave launch most CTAs pass the wait
// at once and the prefetch would just double their L2 requests.
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// Warm L2 with `bytes` contiguous bytes through the bulk-copy engine: one instruction for a whole slice, so
// the issuing thread is free at once and no other thread spends issue slots on it. `p` 16-byte aligned,
// `bytes` a multiple of 16 (every row slice of 16-byte vectors is both).
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ------------------------------------------------------------------------------------------ double-float

// An unevaluated sum hi + lo of two fp32 values (about 48 significant bits), built with Knuth's TwoSum.
// Only additions appear, so no FMA contraction can change the result; TwoSum returns the exact rounding
// error in either operand order, which keeps butterfly reductions identical on every lane.
struct DD {
    float hi, lo;
};

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = a + b;
    const float bp = s - a;
    e = (a - (s - bp)) + (b - bp);
}

__device__ __forceinline__ void dd_accumulate(DD& acc, float x) {
    float s, e;
    two_sum(acc.hi, x, s, e);
    acc.hi = s;
    acc.lo += e;
}

// Two independent double-float accumulators advanced with packed fp32x2 additions (lanes x and y).
struct DD2 {
    float2 hi, lo;
};

__device__ __forceinline__ void dd_accumulate(DD2& acc, float2 x) {
    const float2 s = __fadd2_rn(acc.hi, x);
    const float2 bp = __fadd2_rn(s, make_float2(-acc.hi.x, -acc.hi.y));
    const float2 t = __fadd2_rn(s, make_float2(-bp.x, -bp.y));
    const float2 e = __fadd2_rn(__fadd2_rn(acc.hi, make_float2(-t.x, -t.y)), __fadd2_rn(x, make_float2(-bp.x, -bp.y)));
    acc.hi = s;
    acc.lo = __fadd2_rn(acc.lo, e);
}

// Round the double-float pair (hi + lo) in each lane to bf16 as if it were exact: renormalise so that
// hi = fl(hi + lo), then, if hi sits exactly on a bf16 rounding boundary (low 16 bits 0x8000), move it one
// fp32 ulp toward lo. A value off the boundary rounds the same with or without lo.
__device__ __forceinline__ float dd_nudge_bf16(float hi, float lo) {
    const float s = hi + lo;
    const float e = lo - (s - hi);   // exact remainder (|lo| small against hi)
    uint32_t bits = __float_as_uint(s);
    if ((bits & 0xFFFFu) == 0x8000u && e != 0.0f && s != 0.0f) bits += ((e > 0.0f) == (s > 0.0f)) ? 1u : 0xFFFFFFFFu;
    return __uint_as_float(bits);
}

__device__ __forceinline__ DD dd_add(DD a, DD b) {
    float s, e;
    two_sum(a.hi, b.hi, s, e);
    e += a.lo + b.lo;
    const float hi = s + e;
    return DD{hi, e - (hi - s)};
}

// Row statistics of the dynamic-scale norm: the sum of squares as a double-float and max |w * s|.
struct RowStats {
    DD sum_sq;
    float pmax;
    __device__ __forceinline__ static RowStats combine(RowStats a, RowStats b);
    __device__ __forceinline__ RowStats shfl_xor(int o) const {
        return RowStats{DD{__shfl_xor_sync(0xffffffffu, sum_sq.hi, o), __shfl_xor_sync(0xffffffffu, sum_sq.lo, o)},
                        __shfl_xor_sync(0xffffffffu, pmax, o)};
    }
    __device__ __forceinline__ float4 pack() const { return make_float4(sum_sq.hi, sum_sq.lo, pmax, 0.0f); }
    __device__ __forceinline__ static RowStats unpack(float4 f) { return RowStats{DD{f.x, f.y}, f.z}; }
    __device__ __forceinline__ static RowStats zero() { return RowStats{DD{0.0f, 0.0f}, 0.0f}; }
};

__device__ __forceinline__ RowStats RowStats::combine(RowStats a, RowStats b) {
    return RowStats{dd_add(a.sum_sq, b.sum_sq), fmaxf(a.pmax, b.pmax)};
}

}  // namespace mbd
