// Internal interface between the C-ABI layer (api.cu) and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mbd {

// Output variant of a fused kernel.
enum Epilogue : int { kBf16 = 0, kFp8Static = 1, kFp8Dynamic = 2 };

// How one launch covers the [rows, nvec] problem (nvec = row width / 8, one 16-byte bf16 vector each):
// every row is split into `ctas_per_row` slices of `slice` vectors (the last may be shorter), one CTA per
// slice; a CTA of `threads` threads gives each thread up to `vpt` vectors strided by `threads`.
// If the epilogue reduces over the row and ctas_per_row > 1, the CTAs of a row form one thread-block
// cluster and combine their partial results through distributed shared memory.
struct RowPlan {
    int ctas_per_row;
    int slice;
    int threads;
    int vpt;       // 1, 2, 4 or 8
    int prefetch;  // 1: single-wave launch, warm L2 with the inputs before waiting on the previous kernel
};


constexpr int kMaxPartials = 8;

struct NormParams {
    const void* x;                          // unused when n_partials > 0
    const void* partials[kMaxPartials];     // x = bf16(sum of the n_partials tensors) when n_partials > 0
    int n_partials;
    void* residual;
    const void* weight;
    void* out;       // bf16 [T, H] or uint8 codes [T, H]
    float* scale;    // static: [1] read; dynamic: [T] written; unused for bf16
    int64_t rows;
    int nvec;
    int hidden;
    float eps;
};

struct SwigluParams {
    const void* gate_up;
    void* out;       // bf16 [T, I] or uint8 codes [T, I]
    float* scale;
    int64_t rows;
    int nvec;        // I / 8
};

// Launchers: return the cudaError_t of the launch (cudaSuccess when enqueued). Every launch enables
// programmatic stream serialization; the kernels wait on the previous grid before touching memory.
cudaError_t launch_add_rmsnorm(const NormParams& p, Epilogue ep, const RowPlan& plan, cudaStream_t s);
cudaError_t launch_swiglu(const SwigluParams& p, Epilogue ep, const RowPlan& plan, cudaStream_t s);

// Read (and optionally clear) the device error word of each kernel translation unit (synchronous).
cudaError_t device_error_flags_norm(unsigned int* flags, bool clear);
cudaError_t device_error_flags_swiglu(unsigned int* flags, bool clear);
cudaError_t device_error_flags_selftest(unsigned int* flags, bool clear);

// Launch the bounded-wait self-test kernel (one warp).
cudaError_t launch_bounded_wait_probe(long long limit_cycles, cudaStream_t s);

// Fill a launch configuration: grid/block, the cluster attribute when cluster > 1, and PDL.
inline void fill_launch(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, int64_t ctas, int threads,
                        int cluster, cudaStream_t s) {
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
}

}  // namespace mbd
