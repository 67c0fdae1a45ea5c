// Per-slice body of the fused residual add + RMSNorm (bf16, FP8 E4M3 or NVFP4 out; optionally fed by
// partial activations), shared by the one-launch-per-call kernels (norm.cu) and the persistent program
// kernel (program.cu).
#pragma once

#include "common.cuh"
#include "launch.h"

namespace mbd {

struct NormSmem {
    PSum part_sum[32];
    RowStats part_stats[32];
    Exchange ex;
    float row_const[2];
    int ok_flag;
};

namespace {

// Exact fp32 products of the bf16 halves of two packed words by the mixed-precision fma (bf16 operands, fp32
// addend and result): a product of two bf16 values is exact in fp32 and the -0 addend keeps the sign of a zero
// product, so these are the values of unpacking both words and multiplying in fp32, without the unpacking.
__device__ __forceinline__ float2 mul_bf16x2(uint32_t a, uint32_t b) {
    float lo, hi;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, 0f80000000;\n\tfma.rn.f32.bf16 %1, ah, bh, 0f80000000;\n\t}"
        : "=f"(lo), "=f"(hi) : "r"(a), "r"(b));
    return make_float2(lo, hi);
}

// bf16(a + b) for both halves by the packed bf16 add, which rounds the exact sum once. Rounding the fp32 sum gives
// the same bits: that sum is exact unless the addends' exponents differ by 16 or more, and then the smaller one is
// below 2^-15 of the larger, far inside half a bf16 step of it, so both roundings return the larger.
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// acc + a for both bf16 halves of a, one rounding each: the fp32 add of the unpacked values (mixed-precision add).
__device__ __forceinline__ float2 add_f32_bf16x2(float2 acc, uint32_t a) {
    asm("{\n\t.reg .b16 al, ah;\n\tmov.b32 {al, ah}, %2;\n\t"
        "add.rn.f32.bf16 %0, al, %0;\n\tadd.rn.f32.bf16 %1, ah, %1;\n\t}"
        : "+f"(acc.x), "+f"(acc.y) : "r"(a));
    return acc;
}

// acc + a * a for both bf16 halves of a, one rounding each: the fp32 fma of the unpacked values.
__device__ __forceinline__ float2 fma_sq_bf16x2(uint32_t a, float2 acc) {
    float lo, hi;
    asm("{\n\t.reg .b16 al, ah;\n\tmov.b32 {al, ah}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, al, %3;\n\tfma.rn.f32.bf16 %1, ah, ah, %4;\n\t}"
        : "=f"(lo), "=f"(hi) : "r"(a), "f"(acc.x), "f"(acc.y));
    return make_float2(lo, hi);
}

// Quantise y = p * (c_hi + c_lo) to E4M3, rounding the double-float product as if it were exact.
// p * c_hi is split exactly into y_hi + err (FMA); y_lo = err + p * c_lo. Rounding y_hi alone is correct
// unless y_hi lands exactly on a rounding boundary of the E4M3 grid; every such boundary (and every code
// value) has its 19 low fp32 mantissa bits clear, so a value of that form is moved one fp32 ulp toward
// y_hi + y_lo. A one-ulp move cannot cross a boundary that y_hi was not already on.
__device__ __forceinline__ float nudge(float y_hi, float y_lo) {
    uint32_t bits = __float_as_uint(y_hi);
    if ((bits & 0x7FFFFu) == 0u && y_lo != 0.0f && y_hi != 0.0f) bits += ((y_lo > 0.0f) == (y_hi > 0.0f)) ? 1u : 0xFFFFFFFFu;
    return __uint_as_float(bits);
}

__device__ __forceinline__ float2 exact_side(float2 p, float c_hi, float c_lo) {
    const float2 y_hi = __fmul2_rn(p, f2(c_hi));
    const float2 y_lo = __ffma2_rn(p, f2(c_lo), __ffma2_rn(p, f2(c_hi), make_float2(-y_hi.x, -y_hi.y)));
    return make_float2(nudge(y_hi.x, y_lo.x), nudge(y_hi.y, y_lo.y));
}

// Sum the partial activations of one vector and round once to bf16, as the exact sum rounds: the reduced
// activation x of the all-reduce half. The CTA's slices of the n partials sit in shared memory (brought in by
// bulk copies, `slice` vectors each, this thread's vector at index c of every slice).
//
// Fast path: the plain fp32 sum s (from +0, each partial's bf16 halves added by the mixed-precision add) is exact
// when the addends' exponents span little.
// Every addend is a multiple of 2^(emin - 134) (emin, emax: the smallest and largest bf16 exponent field
// among the element's addends, read off the smallest and largest magnitude; a field of 0, a zero or a
// subnormal, is the conservative case) and every partial sum is below k 2^(emax - 126) <= 2^(emax - 126 + L),
// L = ceil(log2 k); fp32 holds every multiple of that step below 2^24 times it, so each addition is exact when
// emax - emin <= 16 - L, and s is then the exact sum. Elements with a wider span are summed again exactly from
// shared memory (a double-float sum, Knuth's TwoSum, rounded by dd_nudge_bf16), element slot by element slot,
// so a warp runs a slot's exact sum only when one of its lanes needs it (about 1 element in 1000 of N(0,1)
// partials, k = 8).
__device__ __forceinline__ uint4 reduce_partials_smem(const uint4* slices, int slice, int n, int c) {
    float2 s[4];
    uint32_t emax[4], emin[4];   // largest and smallest addend magnitude, lane by lane (bf16 bits)
    {
        const uint4 v = slices[c];
        const uint32_t* w = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            s[q] = add_f32_bf16x2(f2(0.0f), w[q]);   // from +0, as the exact sum: -0 + -0 is +0
            emax[q] = emin[q] = w[q] & 0x7FFF7FFFu;
        }
    }
#pragma unroll
    for (int k = 1; k < kMaxPartials; ++k) {
        if (k >= n) break;
        const uint4 v = slices[k * slice + c];
        const uint32_t* w = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            s[q] = add_f32_bf16x2(s[q], w[q]);
            const uint32_t m = w[q] & 0x7FFF7FFFu;
            emax[q] = max_bf16x2_bits(emax[q], m);
            emin[q] = min_bf16x2_bits(emin[q], m);
        }
    }
    // largest exact span, in exponent-field units at bit 7: 16 - ceil(log2 n)
    const uint32_t span_max = static_cast<uint32_t>(n <= 1 ? 16 : (n <= 2 ? 15 : (n <= 4 ? 14 : 13))) << 7;
    unsigned int redo = 0;   // bit e: element e must be summed exactly
    uint4 x;
    uint32_t* xw = reinterpret_cast<uint32_t*>(&x);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t span = (emax[q] & 0x7F807F80u) - (emin[q] & 0x7F807F80u);   // lane-wise: no borrow
        if ((span & 0xFFFFu) > span_max) redo |= 1u << (2 * q);
        if ((span >> 16) > span_max) redo |= 2u << (2 * q);
        xw[q] = pack_bf16x2(s[q]);
    }
    if (redo) {
        const uint16_t* e16 = reinterpret_cast<const uint16_t*>(slices);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            if (!(redo & (1u << e))) continue;
            DD acc{0.0f, 0.0f};
            for (int k = 0; k < n; ++k)
                dd_accumulate(acc, __uint_as_float(static_cast<uint32_t>(e16[(k * slice + c) * 8 + e]) << 16));
            const float v = dd_nudge_bf16(acc.hi, acc.lo);
            const uint32_t b16 = pack_bf16x2(v, 0.0f) & 0xFFFFu;
            xw[e >> 1] = (e & 1) ? ((xw[e >> 1] & 0x0000FFFFu) | (b16 << 16)) : ((xw[e >> 1] & 0xFFFF0000u) | b16);
        }
    }
    return x;
}

// Thread 0: the CTA's slices of the n partials, `slice` vectors each from vector `begin` of `row` (`count` of them
// are real), into shared memory by bulk copies counted on the mbarrier `bar` (initialised beforehand).
__device__ __forceinline__ void load_partials_bulk(const NormParams& p, int64_t row, int begin, int count, int slice,
                                                   uint4* slices, uint32_t bar) {
    const uint32_t bytes = static_cast<uint32_t>(count) * 16u;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes * p.n_partials)
                 : "memory");
    for (int k = 0; k < p.n_partials; ++k) {
        const uint4* src = static_cast<const uint4*>(p.partials[k]) + row * p.nvec + begin;
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     ::"r"(smem_addr(slices + k * slice)), "l"(src), "r"(bytes), "r"(bar) : "memory");
    }
}

// Every thread: wait (bounded) for the bulk copies counted on `bar` (phase 0). On expiry: an error bit, and a
// second bounded wait for the copies, which write into this CTA's shared memory, before it may leave.
__device__ __forceinline__ bool wait_partials(uint32_t bar) {
    const long long t0 = clock64();
    uint32_t done = 0;
    while (true) {
        asm volatile("{\n .reg .pred q;\n mbarrier.try_wait.parity.shared::cta.b64 q, [%1], 0;\n selp.u32 %0, 1, 0, q;\n}"
                     : "=r"(done) : "r"(bar) : "memory");
        if (done || clock64() - t0 > kWaitLimitCycles) break;
    }
    if (done) return true;
    if (threadIdx.x == 0) atomicOr(&g_device_error_flags, kDevErrExchangeTimeout);
    const long long t1 = clock64();
    while (!done && clock64() - t1 < kWaitLimitCycles)
        asm volatile("{\n .reg .pred q;\n mbarrier.try_wait.parity.shared::cta.b64 q, [%1], 0;\n selp.u32 %0, 1, 0, q;\n}"
                     : "=r"(done) : "r"(bar) : "memory");
    return false;
}

}  // namespace

// Warm L2 with this thread's vectors of one row slice (inputs only: residual, x or the partials).
template <int VPT, bool ALLRED>
__device__ __forceinline__ void norm_prefetch(const NormParams& p, int64_t row, int begin, int end) {
    const uint4* xr = static_cast<const uint4*>(p.x) + row * p.nvec;
    const uint4* rr = static_cast<const uint4*>(p.residual) + row * p.nvec;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int c = begin + threadIdx.x + i * blockDim.x;
        if (c >= end) continue;
        prefetch_l2(rr + c);
        if constexpr (!ALLRED) prefetch_l2(xr + c);   // the partials come by bulk copies after the wait
    }
}

// Step 3 of the norm for the bf16, static-FP8 and NVFP4 epilogues: v = (w * s) * inv (w * s of two bf16
// values is exact in fp32) and its store, for this thread's vectors of one row slice starting at `begin`.
// SCALE_IN: the static or tensor scale was loaded earlier (`scale_in`), else it is loaded here.
template <int VPT, int EP, bool SCALE_IN = false>
__device__ __forceinline__ void norm_store(const NormParams& p, int64_t row, int begin, const uint4 (&sv)[VPT],
                                           const uint4 (&wv)[VPT], const bool (&live)[VPT], float inv,
                                           float scale_in = 0.0f) {
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
                ow[k] = pack_bf16x2(__fmul2_rn(mul_bf16x2(sw[k], ww[k]), f2(inv)));
            store_stream(outr + (begin + threadIdx.x + i * blockDim.x), o);
        }
    } else if constexpr (EP == kNvfp4) {
        // NVFP4: block scales over 16 elements (this vector and the neighbouring lane's), E2M1 codes of
        // v = (w * s) * inv scaled by the block's decoded scale times the tensor scale.
        const Nvfp4Row nr = nvfp4_row(inv, SCALE_IN ? nvfp4_tensor_scale_of(scale_in) : nvfp4_tensor_scale(p.scale));
        unsigned int* qr = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(p.out) + row * (int64_t)p.nvec * 4);
        uint8_t* sfr = p.out_sf + row * (int64_t)(p.nvec / 2);
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            float2 y[4];
            const uint32_t* sw = reinterpret_cast<const uint32_t*>(&sv[i]);
            const uint32_t* ww = reinterpret_cast<const uint32_t*>(&wv[i]);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                y[k] = live[i] ? mul_bf16x2(sw[k], ww[k]) : f2(0.0f);
            uint32_t sf;
            const uint32_t q = nvfp4_encode(y, nr, &sf);   // whole warp (block max by shuffle)
            if (!live[i]) continue;
            const int c = begin + threadIdx.x + i * blockDim.x;
            store_stream(qr + c, q);
            if ((threadIdx.x & 1) == 0) sfr[c >> 1] = static_cast<uint8_t>(sf);
        }
    } else {
        // static per-tensor scale: codes of v / scale
        const float sc = SCALE_IN ? scale_in : __ldg(p.scale);
        const float c = sc > 0.0f ? inv * (1.0f / sc) : 0.0f;
        uint2* outr = reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.out) + row * (int64_t)p.nvec * 8);
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            if (!live[i]) continue;
            const uint32_t* sw = reinterpret_cast<const uint32_t*>(&sv[i]);
            const uint32_t* ww = reinterpret_cast<const uint32_t*>(&wv[i]);
            float2 y[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                y[k] = __fmul2_rn(mul_bf16x2(sw[k], ww[k]), f2(c));
            store_stream(outr + (begin + threadIdx.x + i * blockDim.x),
                         make_uint2(pack_e4m3x4(y[0], y[1]), pack_e4m3x4(y[2], y[3])));
        }
    }
}

// One CTA's share of one row: vectors [begin, end) of `row` (at most VPT per thread), the CTA being `rank`
// of the `nctas` CTAs of the row (one thread-block cluster when nctas > 1). Every thread of the CTA calls
// it. On a cluster-exchange timeout the CTA returns without writing its outputs. CL: kRowInCta (nctas is 1)
// or kRowInCluster (nctas > 1) compile only the reduction that runs (code for the other, even untaken, has
// cost the kernels about 1%); kRowAny decides at run time.
//
// EARLY_SCALE: where the weight is loaded up front, load the static or tensor scale with it (the single-call
// kernels; the persistent program keeps its register budget for its own prefetches and loads it late).
template <int VPT, int EP, bool ALLRED, int CL = kRowAny, bool EARLY_SCALE = false>
__device__ __forceinline__ void norm_row_slice(const NormParams& p, int64_t row, int rank, int nctas, int begin,
                                               int end, NormSmem& sm, const uint4* pslices = nullptr,
                                               int pslice = 0, uint32_t pbar = 0) {
    PSum* part_sum = sm.part_sum;
    RowStats* part_stats = sm.part_stats;
    Exchange& ex = sm.ex;
    float* row_const = sm.row_const;
    // The weight is an L2 hit; load it up front when registers allow (small rows, latency-bound), else
    // after the reduction. The dynamic variant needs it before the reduction anyway. With it (EARLY_SCALE), the
    // static or tensor scale: otherwise its L2 round trip sits alone between the reduction and the stores.
    constexpr bool kEarlyWeight = EP == kFp8Dynamic || VPT <= 2;
    constexpr bool kEarlyScale = EARLY_SCALE && kEarlyWeight && (EP == kFp8Static || EP == kNvfp4);
    const int ctas_per_row = CL == kRowInCta ? 1 : nctas;
    const bool single = CL == kRowInCta || (CL == kRowAny && nctas == 1);

    const uint4* xr = static_cast<const uint4*>(p.x) + row * p.nvec;
    uint4* rr = static_cast<uint4*>(p.residual) + row * p.nvec;
    const uint4* wr = static_cast<const uint4*>(p.weight);

    // 1. one pass over HBM: x and residual in, s = bf16(x + r) kept packed in registers and written back
    uint4 sv[VPT], wv[VPT];
    float qscale = 0.0f;   // kEarlyScale: the static or tensor scale
    bool live[VPT];
    bool landed = true;   // all-reduce half: the partials' bulk copies completed (false: a bounded wait expired)
    {
        uint4 xv[VPT];
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int c = begin + threadIdx.x + i * blockDim.x;
            live[i] = c < end;
            if (live[i]) {
                if constexpr (!ALLRED) xv[i] = load_stream(xr + c);
                sv[i] = load_stream(rr + c);
                if constexpr (kEarlyWeight && !ALLRED) wv[i] = load_cached(wr + c);
            }
        }
        if constexpr (kEarlyScale) qscale = __ldg(p.scale);
        if constexpr (ALLRED) {
            // the partials' slices are in flight into shared memory (bulk copies issued at kernel start); the
            // barrier that follows makes the copies' mbarrier initialisation visible to every thread
            if (single) __syncthreads(); else exchange_init(ex, ctas_per_row);
            landed = wait_partials(pbar);
#pragma unroll
            for (int i = 0; i < VPT; ++i)
                if (live[i]) xv[i] = reduce_partials_smem(pslices, pslice, p.n_partials, threadIdx.x + i * blockDim.x);
            // the weight only now: issued with the residual loads it would share the small L1 share of this form
            // (the largest shared-memory carveout) with them (measured 2.6% slower at k 8, T 2048, H 16384)
            if constexpr (kEarlyWeight) {
#pragma unroll
                for (int i = 0; i < VPT; ++i)
                    if (live[i]) wv[i] = load_cached(wr + (begin + threadIdx.x + i * blockDim.x));
            }
        } else {
            if (!single) exchange_init(ex, ctas_per_row);   // overlaps the loads in flight
        }
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            if (!live[i] || !landed) continue;
            const uint32_t* xw = reinterpret_cast<const uint32_t*>(&xv[i]);
            uint32_t* sw = reinterpret_cast<uint32_t*>(&sv[i]);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                // the same bits either way; the packed add measured faster in the all-reduce half (1 to 3%) and
                // slower in some decode-size single calls (static FP8, H 16384, T 16: 2.29 -> 2.54 us)
                if constexpr (ALLRED) sw[k] = add_bf16x2(xw[k], sw[k]);
                else sw[k] = pack_bf16x2(__fadd2_rn(bf16x2_to_float2(xw[k]), bf16x2_to_float2(sw[k])));
            }
            store_stream(rr + (begin + threadIdx.x + i * blockDim.x), sv[i]);
        }
    }

    if constexpr (EP != kFp8Dynamic) {
        // 2. sum of squares (fp32) -> inv = 1 / sqrt(mean + eps)
        float2 ss2 = f2(0.0f);
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            if (!live[i]) continue;
            const uint32_t* sw = reinterpret_cast<const uint32_t*>(&sv[i]);
#pragma unroll
            for (int k = 0; k < 4; ++k) ss2 = fma_sq_bf16x2(sw[k], ss2);
        }
        float inv;
        if (single) {   // the whole row in this CTA: one barrier, every thread forms inv
            const PSum t = block_total(PSum{ss2.x + ss2.y}, part_sum);
            inv = 1.0f / sqrtf(t.v / static_cast<float>(p.hidden) + p.eps);
        } else {
            if (!row_reduce(PSum{ss2.x + ss2.y}, part_sum, ex, rank, ctas_per_row, &sm.ok_flag, [&](PSum t) {
                    row_const[0] = 1.0f / sqrtf(t.v / static_cast<float>(p.hidden) + p.eps);
                }))
                return;
            inv = row_const[0];
        }

        if constexpr (!kEarlyWeight) {
#pragma unroll
            for (int i = 0; i < VPT; ++i)
                if (live[i]) wv[i] = load_cached(wr + (begin + threadIdx.x + i * blockDim.x));
        }
        if (!landed) return;   // the error bit is set; nothing is written

        norm_store<VPT, EP, kEarlyScale>(p, row, begin, sv, wv, live, inv, qscale);
    } else {
        // Dynamic per-token scale. The codes are ratios of exact bf16 products, 448 * (w_j s_j) / (w_k s_k),
        // rescaled by the fp32 rounding of the scale, so exact E4M3 ties are common; resolving them as the
        // fp64 definition does needs the row constants to ~1e-13: the sum of squares is kept as a
        // double-float, the per-row constants are formed in fp64 once per CTA, and every element is scaled
        // with a double-float multiplier.
        DD2 acc{f2(0.0f), f2(0.0f)};
        float pmax = 0.0f;
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            if (!live[i]) continue;
            const uint32_t* sw = reinterpret_cast<const uint32_t*>(&sv[i]);
            const uint32_t* ww = reinterpret_cast<const uint32_t*>(&wv[i]);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                dd_accumulate(acc, mul_bf16x2(sw[k], sw[k]));   // exact squares of bf16 values
                const float2 p2 = mul_bf16x2(sw[k], ww[k]);
                pmax = fmaxf(pmax, fmaxf(fabsf(p2.x), fabsf(p2.y)));
            }
        }
        const RowStats mine{dd_add(DD{acc.hi.x, acc.lo.x}, DD{acc.hi.y, acc.lo.y}), pmax};
        if (!row_reduce(mine, part_stats, ex, rank, ctas_per_row, &sm.ok_flag, [&](RowStats st) {
                const double mean_sq = (static_cast<double>(st.sum_sq.hi) + static_cast<double>(st.sum_sq.lo)) /
                                       static_cast<double>(p.hidden);
                const double inv = 1.0 / sqrt(mean_sq + static_cast<double>(p.eps));
                const float sc = static_cast<float>(static_cast<double>(st.pmax) * inv / 448.0);
                const double c = sc > 0.0f ? inv / static_cast<double>(sc) : 0.0;
                const float c_hi = static_cast<float>(c);
                row_const[0] = c_hi;
                row_const[1] = static_cast<float>(c - static_cast<double>(c_hi));
                if (rank == 0 && landed) p.scale[row] = sc;
            }))
            return;
        if (!landed) return;   // the error bit is set; nothing is written
        const float c_hi = row_const[0], c_lo = row_const[1];
        uint2* outr = reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.out) + row * (int64_t)p.nvec * 8);
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            if (!live[i]) continue;
            const uint32_t* sw = reinterpret_cast<const uint32_t*>(&sv[i]);
            const uint32_t* ww = reinterpret_cast<const uint32_t*>(&wv[i]);
            float2 y[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                y[k] = exact_side(mul_bf16x2(sw[k], ww[k]), c_hi, c_lo);
            store_stream(outr + (begin + threadIdx.x + i * blockDim.x),
                         make_uint2(pack_e4m3x4(y[0], y[1]), pack_e4m3x4(y[2], y[3])));
        }
    }
}

}  // namespace mbd
