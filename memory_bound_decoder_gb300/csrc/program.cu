// Persistent program kernel: a list of fused norm / SwiGLU ops in one launch.
//
// Every op maps row t of its inputs to row t of its outputs, so a list of ops can run row by row: ops that
// share a buffer (the residual that consecutive norms update, an output read in place later) form a chain,
// and one CTA runs a chain's ops on one row in list order, with a CTA barrier between ops so that each op
// sees the previous op's stores; no grid-wide synchronisation and no scratch memory are needed. Ops that
// share nothing are split into (row, chunk) items spread over the other CTAs. The per-row arithmetic is the
// same device code as the one-launch-per-call kernels (norm_row_slice, swiglu_row_slice), with the whole
// row in one CTA (no cluster).
//
// This is the launch-overhead remedy in kernel form ("TensorRT-LLM: Compiling Inference Engines Ahead of
// Time", "Fusing operations, measured" and "Leaving the engine behind": issuing many small kernels costs
// more than running them, hence CUDA graphs for decoding; "Introduction to torch.compile and How It Works
// with vLLM", section 5: one kernel for a whole forward pass).
#include <cstddef>
#include <mutex>

#include "norm_impl.cuh"
#include "swiglu_impl.cuh"

namespace mbd {

namespace {

struct ProgSmem {
    NormSmem norm;
    SwigluSmem swiglu;
    alignas(16) PSum run_part[2][32];   // norm_run's warp partials, alternating between consecutive ops
};

// Epilogue sets of a program kernel variant: bit e set = epilogue e compiled in. Each variant carries only
// the epilogues it can meet, which keeps its registers near those of the one-launch-per-call kernels.
constexpr int bit(int ep) { return 1 << ep; }

// The mixed variant's epilogues: bf16 and FP8 ops in one program. The dynamic-FP8 norm (its exact
// double-float scaling) stays out of it.
constexpr int kMixedNormMask = bit(kBf16) | bit(kFp8Static);
constexpr int kMixedSwigluMask = bit(kBf16) | bit(kFp8Static) | bit(kFp8Dynamic);

// Whether a variant runs each row op as a call (__noinline__) instead of inline. Inlined, every op path of
// the mixed variant and of the 8-vectors-per-thread variants shares one register allocation, and they
// spilled 2.5 to 5.4 KB per thread; as calls each path gets its own. The bf16, FP8 and NVFP4 decode variants
// stay inline: a call per row op cost their chained decode programs 20 to 33%.
constexpr bool outlined(int v, int nm, int sm) { return v == 8 || (nm == kMixedNormMask && sm == kMixedSwigluMask); }

// The wide form (V = 8 in the templates: a row of up to kProgramThreads * 8 vectors in one CTA) runs
// kProgramWideThreads threads. Its norm rows (at most kProgramThreads * 4 vectors, MBD_MAX_PROGRAM_WIDTH) and
// stream chunks (kProgramThreads * 4 vectors) take one vector per thread, its dynamic-FP8 SwiGLU rows two.
constexpr int threads_of(int v) { return v == 8 ? kProgramWideThreads : kProgramThreads; }
constexpr int held_vpt(int v) { return v == 8 ? kProgramThreads * 8 / kProgramWideThreads : v; }
constexpr int chunk_vpt(int v) { return v == 8 ? kProgramThreads * 4 / kProgramWideThreads : v; }
static_assert(kProgramThreads * 8 % kProgramWideThreads == 0 && kProgramThreads * 4 % kProgramWideThreads == 0,
              "the wide form holds whole vectors per thread");

template <int V8, int NM>
__device__ __forceinline__ void run_norm_row(const ProgOp& op, int64_t row, ProgSmem& sm) {
    constexpr int V = chunk_vpt(V8);
    NormParams np;
    np.x = op.in;
    np.n_partials = 0;
    np.residual = op.residual;
    np.weight = op.weight;
    np.out = op.out;
    np.out_sf = op.out_sf;
    np.scale = op.scale;
    np.rows = op.rows;
    np.nvec = op.nvec;
    np.hidden = op.hidden;
    np.eps = op.eps;
    if constexpr ((NM & bit(kBf16)) != 0) {
        if (op.ep == kBf16) return norm_row_slice<V, kBf16, false, kRowInCta>(np, row, 0, 1, 0, op.nvec, sm.norm);
    }
    if constexpr ((NM & bit(kFp8Static)) != 0) {
        if (op.ep == kFp8Static) return norm_row_slice<V, kFp8Static, false, kRowInCta>(np, row, 0, 1, 0, op.nvec, sm.norm);
    }
    if constexpr ((NM & bit(kFp8Dynamic)) != 0) {
        if (op.ep == kFp8Dynamic) return norm_row_slice<V, kFp8Dynamic, false, kRowInCta>(np, row, 0, 1, 0, op.nvec, sm.norm);
    }
    if constexpr ((NM & bit(kNvfp4)) != 0) {
        if (op.ep == kNvfp4) return norm_row_slice<V, kNvfp4, false, kRowInCta>(np, row, 0, 1, 0, op.nvec, sm.norm);
    }
}

// Vectors [begin, end) of one SwiGLU row (a stream chunk: end - begin <= kProgramThreads * min(V8, 4); the
// whole row for the dynamic epilogue, which reduces over it, when it fits kProgramThreads * V8).
template <int V8, int SM>
__device__ __forceinline__ void run_swiglu_part(const ProgOp& op, int64_t row, int begin, int end, ProgSmem& sm) {
    constexpr int V = chunk_vpt(V8);
    SwigluParams sp{op.in, op.out, op.scale, op.rows, op.nvec, op.out_sf};
    if constexpr ((SM & bit(kBf16)) != 0) {
        if (op.ep == kBf16) return swiglu_row_slice<V, kBf16, kRowInCta>(sp, row, 0, 1, begin, end, sm.swiglu);
    }
    if constexpr ((SM & bit(kFp8Static)) != 0) {
        if (op.ep == kFp8Static) return swiglu_row_slice<V, kFp8Static, kRowInCta>(sp, row, 0, 1, begin, end, sm.swiglu);
    }
    if constexpr ((SM & bit(kFp8Dynamic)) != 0) {
        if (op.ep == kFp8Dynamic) return swiglu_row_slice<held_vpt(V8), kFp8Dynamic, kRowInCta>(sp, row, 0, 1, begin, end, sm.swiglu);
    }
    if constexpr ((SM & bit(kNvfp4)) != 0) {
        if (op.ep == kNvfp4) return swiglu_row_slice<V, kNvfp4, kRowInCta>(sp, row, 0, 1, begin, end, sm.swiglu);
    }
}

// A dynamic FP8 SwiGLU row: one pass from registers when it fits the CTA (kProgramThreads * V vectors),
// else two passes (max, then codes).
template <int V, int SM>
__device__ __forceinline__ void run_swiglu_dynamic_row(const ProgOp& op, int64_t row, ProgSmem& sm) {
    if constexpr ((SM & bit(kFp8Dynamic)) != 0) {
        if (op.nvec <= kProgramThreads * V) return run_swiglu_part<V, SM>(op, row, 0, op.nvec, sm);
        SwigluParams sp{op.in, op.out, op.scale, op.rows, op.nvec, op.out_sf};
        // V = 4 (one CTA per SM, registers to spare): 4 vectors per thread in flight per step; else one (few
        // registers at 2 to 4 CTAs per SM, or 1024 threads in the wide form)
        swiglu_dynamic_two_pass<(V == 4 ? 4 : 1)>(sp, row, sm.swiglu);
    }
}

// Out-of-line forms of the row-op runners (see outlined()).
template <int V, int NM>
__device__ __noinline__ void run_norm_row_call(const ProgOp& op, int64_t row, ProgSmem& sm) {
    run_norm_row<V, NM>(op, row, sm);
}
template <int V, int SM>
__device__ __noinline__ void run_swiglu_part_call(const ProgOp& op, int64_t row, int begin, int end, ProgSmem& sm) {
    run_swiglu_part<V, SM>(op, row, begin, end, sm);
}
template <int V, int SM>
__device__ __noinline__ void run_swiglu_dynamic_row_call(const ProgOp& op, int64_t row, ProgSmem& sm) {
    run_swiglu_dynamic_row<V, SM>(op, row, sm);
}

// One row op, inline or as a call: a norm or a dynamic-FP8 SwiGLU on the whole row, or a SwiGLU stream on
// vectors [begin, end) in chunks of `chunk`.
template <int V, int NM, int SM>
__device__ __forceinline__ void run_row_op(const ProgOp& op, int64_t row, int begin, int end, int chunk, ProgSmem& sm) {
    if (op.cls == kOpNorm) {
        if constexpr (outlined(V, NM, SM)) run_norm_row_call<V, NM>(op, row, sm);
        else run_norm_row<V, NM>(op, row, sm);
    } else if (op.ep == kFp8Dynamic) {
        if constexpr (outlined(V, NM, SM)) run_swiglu_dynamic_row_call<V, SM>(op, row, sm);
        else run_swiglu_dynamic_row<V, SM>(op, row, sm);
    } else {
        for (int b = begin; b < end; b += chunk) {
            if constexpr (outlined(V, NM, SM)) run_swiglu_part_call<V, SM>(op, row, b, min(b + chunk, end), sm);
            else run_swiglu_part<V, SM>(op, row, b, min(b + chunk, end), sm);
        }
    }
}

__device__ __forceinline__ void warm_row(const void* base, int64_t row, int nvec) {
    const uint4* r = static_cast<const uint4*>(base) + row * nvec;
    for (int c = threadIdx.x; c < nvec; c += blockDim.x) prefetch_l2(r + c);
}

// The one epilogue a mask holds, or -1.
constexpr int single_ep(int mask) {
    return mask == bit(kBf16) ? kBf16
         : mask == bit(kFp8Static) ? kFp8Static
         : mask == bit(kFp8Dynamic) ? kFp8Dynamic
         : mask == bit(kNvfp4) ? kNvfp4 : -1;
}

// A run of consecutive norms of one chain on the same residual row (the layers of a decode step), ops
// ops[0 .. n), whole rows of one vector per thread. The residual row stays in registers across the run and
// is stored once at its end: the values in between would be overwritten by the next norm of the run, and
// no op outside the chain reads that buffer. The next op's x and weight vectors (which no earlier op of the
// chain writes) are loaded before this op's reduction, so their L2 latency overlaps the reduction and the
// epilogue instead of adding to them.
template <int EP>
__device__ void norm_run(const ProgOp* ops, int n, int64_t row, ProgSmem& sm) {
    const int nvec = ops[0].nvec;
    // every norm of a run has the same width (the planner links only equal widths), so 1 / hidden is
    // formed once: a correctly rounded division per op sat on the chain's critical path
    const float inv_h = 1.0f / static_cast<float>(ops[0].hidden);
    const int c = threadIdx.x;
    const bool live[1] = {c < nvec};
    uint4* rr = static_cast<uint4*>(ops[0].residual) + row * nvec + c;
    uint4 sv[1], xv, wv[1];
    if (live[0]) {
        sv[0] = load_cached(rr);
        xv = load_stream(static_cast<const uint4*>(ops[0].in) + row * nvec + c);
        wv[0] = load_cached(static_cast<const uint4*>(ops[0].weight) + c);
    }
    // static FP8: the op's code multiplier 1 / scale, its scale loaded one op ahead (a global load and a
    // division per op would otherwise sit on the chain)
    float qmul = 0.0f, sc_next = 0.0f;
    if constexpr (EP == kFp8Static) {
        const float sc = __ldg(ops[0].scale);
        qmul = sc > 0.0f ? 1.0f / sc : 0.0f;
    }
    for (int k = 0; k < n; ++k) {
        const ProgOp& op = ops[k];
        float2 ss2 = f2(0.0f);
        if (live[0]) {
            const uint32_t* xw = reinterpret_cast<const uint32_t*>(&xv);
            uint32_t* sw = reinterpret_cast<uint32_t*>(&sv[0]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                sw[q] = add_bf16x2(xw[q], sw[q]);
                ss2 = fma_sq_bf16x2(sw[q], ss2);
            }
        }
        uint4 wn;
        if (k + 1 < n && live[0]) {   // the next op's inputs (x into the spent x registers)
            xv = load_stream(static_cast<const uint4*>(ops[k + 1].in) + row * nvec + c);
            wn = load_cached(static_cast<const uint4*>(ops[k + 1].weight) + c);
        }
        if constexpr (EP == kFp8Static) {
            if (k + 1 < n) sc_next = __ldg(ops[k + 1].scale);
        }
        // Partials alternate between two buffers: when a thread writes op k + 2's partials into this one,
        // every thread has passed op k + 1's barrier and so has read op k's, so no barrier closes the op.
        const PSum t = block_total_tree(PSum{ss2.x + ss2.y}, sm.run_part[k & 1]);
        // the hardware reciprocal square root and a multiply by 1 / hidden instead of a correctly rounded
        // square root and two divisions: a few ulps, against a bf16 tolerance of 2^-7, and a shorter
        // dependent chain on the decode step's critical path
        const float inv = rsqrtf(t.v * inv_h + op.eps);
        if constexpr (EP == kFp8Static) {   // the codes of v / scale, as norm_store forms them
            if (live[0]) {
                const float cm = inv * qmul;
                const uint32_t* sw = reinterpret_cast<const uint32_t*>(&sv[0]);
                const uint32_t* ww = reinterpret_cast<const uint32_t*>(&wv[0]);
                float2 y[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    y[q] = __fmul2_rn(mul_bf16x2(sw[q], ww[q]), f2(cm));
                store_stream(reinterpret_cast<uint2*>(static_cast<uint8_t*>(op.out) + row * (int64_t)nvec * 8) + c,
                             make_uint2(pack_e4m3x4(y[0], y[1]), pack_e4m3x4(y[2], y[3])));
            }
            if (k + 1 < n) qmul = sc_next > 0.0f ? 1.0f / sc_next : 0.0f;
        } else {
            NormParams np;
            np.x = op.in;
            np.n_partials = 0;
            np.residual = op.residual;
            np.weight = op.weight;
            np.out = op.out;
            np.out_sf = op.out_sf;
            np.scale = op.scale;
            np.rows = op.rows;
            np.nvec = op.nvec;
            np.hidden = op.hidden;
            np.eps = op.eps;
            norm_store<1, EP>(np, row, 0, sv, wv, live, inv);
        }
        if (k + 1 < n) wv[0] = wn;
    }
    if (live[0]) store_stream(rr, sv[0]);
}

// A chain CTA's copy of its chain's op descriptors: read in place, every descriptor would be a dynamically
// indexed constant-bank load on the chain's critical path, once per op.
struct ChainSmem {
    ProgOp ops[kMaxProgramOps];
};

template <int V, int NM, int SM>
// `g` is the chain of this item's CTA cursor and `held` the chain whose descriptors cs.ops holds (-1: none);
// both live in registers and every thread of the CTA updates them identically.
__device__ void run_chain_item(const ProgramParams& P, int64_t item, int& g, int& held, ProgSmem& sm, ChainSmem& cs) {
    while (g + 1 < P.n_groups && P.group_items[g + 1] <= item) ++g;   // items of a CTA only increase
    const int64_t row = item - P.group_items[g];
    const int k0 = P.group_begin[g], n = P.group_begin[g + 1] - k0;
    if (held != g) {
        __syncthreads();   // every thread is done with the previous chain's descriptors
        constexpr int kWords = sizeof(ProgOp) / 4;
        for (int w = threadIdx.x; w < n * kWords; w += blockDim.x) {
            const uint32_t* src = reinterpret_cast<const uint32_t*>(&P.ops[P.chain_order[k0 + w / kWords]]);
            reinterpret_cast<uint32_t*>(cs.ops)[w] = src[w % kWords];
        }
        __syncthreads();
        held = g;
    }
    if (P.prefetch_chains) {
        for (int k = 0; k < n; ++k) {
            const ProgOp& op = cs.ops[k];
            const int in_vecs = op.cls == kOpNorm ? op.nvec : 2 * op.nvec;
            if (op.prefetch & 1) warm_row(op.in, row, in_vecs);
            if (op.prefetch & 2) warm_row(op.residual, row, op.nvec);
        }
    }
    for (int k = 0; k < n; ++k) {
        const ProgOp& op = cs.ops[k];
        if constexpr (V == 1 && single_ep(NM) >= 0 && single_ep(NM) != kFp8Dynamic) {
            if (op.cls == kOpNorm) {
                int e = k + 1;
                while (e < n && (cs.ops[e].prefetch & kContinuesRun)) ++e;
                if (e - k > 1) {   // ops k .. e - 1 run with the residual row in registers
                    norm_run<single_ep(NM)>(cs.ops + k, e - k, row, sm);
                    k = e - 1;
                    __syncthreads();
                    continue;
                }
            }
        }
        run_row_op<V, NM, SM>(op, row, 0, op.nvec, P.chunk_vecs, sm);
        __syncthreads();   // this op's stores are visible to every thread before the next op reads them
    }
}

template <int V, int NM, int SM>
__device__ void run_free_item(const ProgramParams& P, int64_t item, int& f, ProgSmem& sm) {
    while (f + 1 < P.n_free && P.free_items[f + 1] <= item) ++f;   // items of a CTA only increase
    const ProgOp& op = P.ops[P.free_op[f]];
    const int64_t local = item - P.free_items[f];
    const int chunks = P.free_chunks[f];
    const int64_t row = local / chunks;
    const int chunk = static_cast<int>(local - row * chunks);
    const int b = chunks == 1 ? 0 : chunk * P.chunk_vecs;
    const int e = chunks == 1 ? op.nvec : min(b + P.chunk_vecs, op.nvec);
    run_row_op<V, NM, SM>(op, row, b, e, P.chunk_vecs, sm);
    __syncthreads();   // the next item's reduction may reuse the warp partials
}

// Resident CTAs per SM each variant is compiled for (the register cap): the most that leaves it without
// large spills, from ptxas -v (40 to 255 registers; a few variants keep spills of under 200 bytes). The FP8 variant at 4 vectors per thread takes the whole
// register file at one CTA per SM: capped at 128 registers for two it spilled 1 to 2.6 KB per thread, and
// its programs ran 1.6x (8 layers at 64 tokens) to 3.9x (at 256 tokens) slower than at one. The wide form
// (1024 threads) is one CTA per SM as well.
constexpr int min_ctas(int v, int nm, int sm) {
    return (sm & bit(kFp8Dynamic)) != 0 ? (v == 1 ? 4 : (v == 2 ? 2 : 1))   // the dynamic SwiGLU's two-pass form adds registers
                                  : (v == 1 ? ((nm == bit(kBf16) && sm == bit(kBf16)) ? 6 : 5) : (v == 2 ? 3 : 2));
}

// Chain items take CTAs 0 .. n_chain - 1 and free items the CTAs after them, so a chain (the critical path
// of a decode step) shares its CTA with nothing; when there are more chain items than CTAs both kinds are
// dealt round-robin over the whole grid.
template <int V, int NM, int SM>
__device__ __forceinline__ void program_body(const ProgramParams& P) {
    __shared__ ProgSmem sm;
    __shared__ ChainSmem cs;
    const int64_t G = gridDim.x, b = blockIdx.x;
    const int64_t nc = P.n_chain_items, nf = P.n_free_items;
    int g = 0, held = -1, f = 0;
    if (nc < G) {
        if (b < nc) {
            run_chain_item<V, NM, SM>(P, b, g, held, sm, cs);
        } else {
            for (int64_t j = b - nc; j < nf; j += G - nc) run_free_item<V, NM, SM>(P, j, f, sm);
        }
    } else {
        for (int64_t i = b; i < nc; i += G) run_chain_item<V, NM, SM>(P, i, g, held, sm, cs);
        for (int64_t j = b; j < nf; j += G) run_free_item<V, NM, SM>(P, j, f, sm);
    }
}

// The schedule by value in the kernel parameters (no device memory needed; a launch carries ~14 KB)...
template <int V, int NM, int SM>
__global__ void __launch_bounds__(threads_of(V), min_ctas(V, NM, SM)) program_kernel(const __grid_constant__ ProgramParams P) {
    pdl_wait();
    program_body<V, NM, SM>(P);
    pdl_trigger();   // late: a dependent program waiting in SM slots would hold resources this one still uses
}

// ... or uploaded by the caller to device memory (a launch carries one pointer). Every CTA first copies the
// used part of it into shared memory with coalesced loads (one L2 round trip), so that the item lookups and
// descriptors cost shared-memory latency rather than an L2 round trip each. The upload precedes the launch
// in stream order and is not a kernel, so the copy may run before the grid dependency wait.
// `order` (PdlOrder): kPdlWaitFirst for a program on its own (wait, run, then let the next kernel start: a
// dependent program waiting in SM slots would hold resources this one still uses); in a batch of independent
// launches (mbd_run_independent_with_program), kPdlHead (wait, let the next launch start, run) or kPdlOverlap
// (let the next launch start, run without waiting, wait for the previous launch before exiting).
template <int V, int NM, int SM>
__global__ void __launch_bounds__(threads_of(V), min_ctas(V, NM, SM)) program_kernel_dev(const ProgramParams* __restrict__ P,
                                                                                        int order) {
    __shared__ __align__(16) ProgramParams S;
    {
        const size_t bytes = offsetof(ProgramParams, ops) + static_cast<size_t>(P->n_ops) * sizeof(ProgOp);
        const int words = static_cast<int>(bytes / 8);
        const uint2* src = reinterpret_cast<const uint2*>(P);
        uint2* dst = reinterpret_cast<uint2*>(&S);
        for (int i = threadIdx.x; i < words; i += blockDim.x) dst[i] = src[i];
    }
    __syncthreads();
    if (order != kPdlOverlap) pdl_wait();
    if (order != kPdlWaitFirst) pdl_trigger();
    program_body<V, NM, SM>(S);
    if (order == kPdlOverlap) pdl_wait();
    pdl_trigger();   // late, as in program_kernel (a no-op after an early one)
}

template <int V, int NM, int SM>
int ctas_per_sm() {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, program_kernel<V, NM, SM>, threads_of(V), 0) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

template <int V, int NM, int SM>
cudaError_t launch_variant(const ProgramParams& p, const ProgramParams* dev, int grid, cudaStream_t s, int order) {
    cudaLaunchConfig_t cfg = cudaLaunchConfig_t{};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(threads_of(V), 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dev) return cudaLaunchKernelEx(&cfg, program_kernel_dev<V, NM, SM>, dev, order);
    return cudaLaunchKernelEx(&cfg, program_kernel<V, NM, SM>, p);
}

// The compiled variants: (norm epilogues, SwiGLU epilogues). A program takes the first that covers its ops.
constexpr int kVariantMasks[kProgramVariants][2] = {
    {bit(kBf16), bit(kBf16)},                  // bf16 layers
    {bit(kFp8Static), bit(kFp8Dynamic)},       // FP8: static-scale norm, dynamic-scale SwiGLU
    {bit(kNvfp4), bit(kNvfp4)},                // NVFP4 layers
    {kMixedNormMask, kMixedSwigluMask},        // bf16 and FP8 ops mixed in one program
};

constexpr bool has_vpt8(int k) { return (kVariantMasks[k][1] & bit(kFp8Dynamic)) != 0; }

template <int V, int K>
int ctas_of() { return ctas_per_sm<V, kVariantMasks[K][0], kVariantMasks[K][1]>(); }

template <int V, int K>
cudaError_t launch_of(const ProgramParams& p, const ProgramParams* dev, int grid, cudaStream_t s, int head) {
    return launch_variant<V, kVariantMasks[K][0], kVariantMasks[K][1]>(p, dev, grid, s, head);
}

template <int V>
int ctas_v(int variant) {
    switch (variant) {
        case 0: return ctas_of<V, 0>();
        case 1: return ctas_of<V, 1>();
        case 2: return ctas_of<V, 2>();
        case 3: return ctas_of<V, 3>();
    }
    return 0;
}

template <int V>
cudaError_t launch_v(const ProgramParams& p, const ProgramParams* dev, int variant, int grid, cudaStream_t s, int head) {
    switch (variant) {
        case 0: return launch_of<V, 0>(p, dev, grid, s, head);
        case 1: return launch_of<V, 1>(p, dev, grid, s, head);
        case 2: return launch_of<V, 2>(p, dev, grid, s, head);
        case 3: return launch_of<V, 3>(p, dev, grid, s, head);
    }
    return cudaErrorInvalidValue;
}

// 8 vectors per thread: compiled only for the variants with the dynamic-FP8 SwiGLU.
static_assert(has_vpt8(1) && has_vpt8(3) && !has_vpt8(0) && !has_vpt8(2), "variants compiled at 8 vectors per thread");

int ctas_v8(int variant) {
    switch (variant) {
        case 1: return ctas_of<8, 1>();
        case 3: return ctas_of<8, 3>();
    }
    return 0;
}

cudaError_t launch_v8(const ProgramParams& p, const ProgramParams* dev, int variant, int grid, cudaStream_t s, int head) {
    switch (variant) {
        case 1: return launch_of<8, 1>(p, dev, grid, s, head);
        case 3: return launch_of<8, 3>(p, dev, grid, s, head);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

int program_variant(int norm_mask, int swiglu_mask) {
    for (int k = 0; k < kProgramVariants; ++k)
        if ((norm_mask & ~kVariantMasks[k][0]) == 0 && (swiglu_mask & ~kVariantMasks[k][1]) == 0) return k;
    return -1;
}

bool program_variant_has_vpt8(int variant) { return variant >= 0 && variant < kProgramVariants && has_vpt8(variant); }

bool program_norms_in_registers(int vpt, int variant) {
    if (variant < 0 || variant >= kProgramVariants) return false;
    const int ep = single_ep(kVariantMasks[variant][0]);
    return vpt == 1 && ep >= 0 && ep != kFp8Dynamic;
}

int program_ctas_per_sm(int vpt, int variant) {
    switch (vpt) {
        case 1: return ctas_v<1>(variant);
        case 2: return ctas_v<2>(variant);
        case 4: return ctas_v<4>(variant);
        case 8: return ctas_v8(variant);
    }
    return 0;
}

cudaError_t launch_program(const ProgramParams& p, const ProgramParams* dev, int vpt, int variant, int grid,
                           cudaStream_t s, int order) {
    if (order != kPdlWaitFirst && !dev) return cudaErrorInvalidValue;   // only the uploaded form joins a batch
    const int h = order;
    switch (vpt) {
        case 1: return launch_v<1>(p, dev, variant, grid, s, h);
        case 2: return launch_v<2>(p, dev, variant, grid, s, h);
        case 4: return launch_v<4>(p, dev, variant, grid, s, h);
        case 8: return launch_v8(p, dev, variant, grid, s, h);
    }
    return cudaErrorInvalidValue;
}

// Schedule storage of mbd_program_plan_launch_static, for callers that cannot allocate device memory: part
// of the module image (every GPU that loads the library holds it until exit), so nothing is allocated when
// it is used. In host code the name is a host-side stand-in, not a device address: the kernel gets the
// address that cudaGetSymbolAddress returns with the device current.
static __device__ __align__(256) unsigned char g_static_schedule[kStaticScheduleBytes];

namespace {
// Per device: the buffer's address and the id of the context it was looked up in. The module's globals live
// in a context; cudaDeviceReset destroys the device's primary context, and the one that replaces it may load
// the module at another address, so an address is reused only while the same context is current.
struct StaticScheduleSlot {
    unsigned long long context = 0;
    void* addr = nullptr;
};
std::mutex g_static_schedule_mu;
StaticScheduleSlot g_static_schedule_slot[kMaxCachedDevices];
}  // namespace

cudaError_t static_schedule_address(int device, void** addr) {
    if (device < 0 || device >= kMaxCachedDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_static_schedule_mu);
    StaticScheduleSlot& slot = g_static_schedule_slot[device];
    const unsigned long long ctx = current_context_id();
    if (ctx != 0 && slot.context == ctx && slot.addr) {
        *addr = slot.addr;
        return cudaSuccess;
    }
    void* a = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&a, g_static_schedule);
    if (e != cudaSuccess) return e;
    if (!a) return cudaErrorInvalidSymbol;
    // The lookup makes the device's primary context current if none was, so its id is read afterwards; with
    // no id (0) the slot never matches and every call looks the address up.
    slot.context = current_context_id();
    slot.addr = a;
    *addr = a;
    return cudaSuccess;
}

cudaError_t device_error_flags_program(unsigned int* flags, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_device_error_flags, sizeof(unsigned int));
    if (e == cudaSuccess && clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error_flags, &zero, sizeof(unsigned int));
    }
    return e;
}

}  // namespace mbd
