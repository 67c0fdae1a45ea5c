// Internal interface between the C-ABI layer (api.cu) and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mbd {

// Output variant of a fused kernel.
enum Epilogue : int { kBf16 = 0, kFp8Static = 1, kFp8Dynamic = 2, kNvfp4 = 3 };

// How one launch covers the [rows, nvec] problem (nvec = row width / 8, one 16-byte bf16 vector each):
// every row is split into `ctas_per_row` slices of `slice` vectors (the last may be shorter), one CTA per
// slice; a CTA of `threads` threads gives each thread up to `vpt` vectors strided by `threads`.
// If the epilogue reduces over the row and ctas_per_row > 1, the CTAs of a row form one thread-block
// cluster and combine their partial results through distributed shared memory. The NVFP4 epilogue needs
// even slices, so that the two vectors of every 16-element block sit in neighbouring lanes of one warp.
struct RowPlan {
    int ctas_per_row;
    int slice;
    int threads;
    int vpt;       // 1, 2, 4 or 8
    int prefetch;  // 1: single-wave launch, warm L2 with the inputs before waiting on the previous kernel
    int ahead;     // > 0: each CTA also warms L2 with the same slice of row + ahead (a later wave's row)
    int bulk;      // dynamic-FP8 SwiGLU: 1 = the slices come into shared memory by bulk copies (vpt 4)
    int order;     // PdlOrder: how the launch orders itself against the previous kernel on the stream
};

// Programmatic dependent launch order of a single-call kernel (RowPlan::order). kPdlWaitFirst for every
// call on its own; a batch of independent ops (mbd_run_independent) launches its first op kPdlHead and the
// rest kPdlOverlap (a later op's CTAs run while the previous op's still do, and wait for it only before they
// exit). Legal only where no op of the batch touches memory that another op of the batch writes.
enum PdlOrder : int { kPdlWaitFirst = 0, kPdlHead = 1, kPdlOverlap = 2 };


constexpr int kMaxPartials = 8;

struct NormParams {
    const void* x;                          // unused when n_partials > 0
    const void* partials[kMaxPartials];     // x = bf16(sum of the n_partials tensors) when n_partials > 0
    int n_partials;
    void* residual;
    const void* weight;
    void* out;       // bf16 [T, H], E4M3 codes [T, H] or packed E2M1 codes [T, H / 2]
    uint8_t* out_sf; // NVFP4 block scales [T, H / 16] (E4M3); unused otherwise
    float* scale;    // FP8 static and NVFP4: [1] read; FP8 dynamic: [T] written; unused for bf16
    int64_t rows;
    int nvec;
    int hidden;
    float eps;
};

struct SwigluParams {
    const void* gate_up;
    void* out;       // bf16 [T, I], E4M3 codes [T, I] or packed E2M1 codes [T, I / 2]
    float* scale;    // as in NormParams
    int64_t rows;
    int nvec;        // I / 8
    uint8_t* out_sf; // NVFP4 block scales [T, I / 16]
};

// ------------------------------------------------------------------------------------------ programs

constexpr int kMaxProgramOps = 128;     // MBD_MAX_PROGRAM_OPS
constexpr int kProgramThreads = 256;    // CTA size of the program kernel
// The wide form (vpt 8 on the host: a row of up to kProgramThreads * 8 vectors held by one CTA) runs
// kProgramWideThreads threads of at most 2 vectors each.
constexpr int kProgramWideThreads = 1024;
constexpr int kMaxProgramGroups = kMaxProgramOps / 2;

enum OpClass : int { kOpNorm = 0, kOpSwiglu = 1 };

// One op of a program, as the kernel sees it.
struct ProgOp {
    const void* in;      // x (norm) or gate_up (SwiGLU)
    void* residual;      // norm
    const void* weight;  // norm
    void* out;
    uint8_t* out_sf;     // NVFP4 block scales
    float* scale;
    int64_t rows;
    int cls;             // OpClass
    int ep;              // Epilogue
    int nvec;            // width / 8
    int hidden;          // width
    float eps;
    int prefetch;        // chain ops: bit 0 warm `in`, bit 1 warm `residual` (row inputs no earlier op writes),
                         // kContinuesRun: a norm on the previous op's residual row whose x no earlier op writes
};

constexpr int kContinuesRun = 4;

// The whole schedule, passed by value as the kernel's parameters (about 14 KB).
// Chain items: (group g, row t) for t < rows of g; the CTA runs every op of g on row t in list order.
// Free items: (free op f, row t, chunk k); ops that hold their row have one chunk per row.
struct ProgramParams {
    int n_ops;                                  // ops[0 .. n_ops) are filled (the kernel copies only those)
    int n_groups;
    int n_free;
    int chunk_vecs;                             // vectors of one stream chunk (kProgramThreads * min(vpt, 4))
    int prefetch_chains;                        // warm each chain row's external inputs first
    int64_t n_chain_items;
    int64_t n_free_items;
    int chain_order[kMaxProgramOps];            // op indices, group by group, each in list order
    int group_begin[kMaxProgramGroups + 1];     // group g: chain_order[group_begin[g] .. group_begin[g + 1])
    int64_t group_items[kMaxProgramGroups + 1]; // prefix sums of the groups' rows
    int free_op[kMaxProgramOps];
    int free_chunks[kMaxProgramOps];            // items per row of free op f
    int64_t free_items[kMaxProgramOps + 1];     // prefix sums of rows * chunks
    ProgOp ops[kMaxProgramOps];
};

// Compiled program-kernel variants, each for a set of norm and SwiGLU epilogues (bit e = Epilogue e).
constexpr int kProgramVariants = 4;
// The first variant that covers the given epilogue sets, or -1.
int program_variant(int norm_mask, int swiglu_mask);
// Whether `variant` is compiled in the wide form, vpt 8 (the variants with the dynamic-FP8 SwiGLU, whose rows
// of up to kProgramThreads * 8 vectors then run in one pass).
bool program_variant_has_vpt8(int variant);
// Whether `variant` at `vpt` runs consecutive chained norms with the residual row in registers (vpt 1 and a
// single norm epilogue other than dynamic FP8).
bool program_norms_in_registers(int vpt, int variant);
static_assert(sizeof(ProgOp) % 8 == 0 && sizeof(ProgramParams) % 8 == 0, "schedules are copied in 8-byte words");

// The library's own schedule buffer (one per device, a static array of the module image), and its address
// on `device`, which must be the current device (0 <= device < kMaxCachedDevices). The address is looked up
// once per device and context: a context re-created on that device (cudaDeviceReset) is looked up again.
constexpr size_t kStaticScheduleBytes = 16384;
static_assert(sizeof(ProgramParams) <= kStaticScheduleBytes, "a schedule fits the static buffer");
constexpr int kMaxCachedDevices = 64;
cudaError_t static_schedule_address(int device, void** addr);

// The unique id (cuCtxGetId) of the calling thread's current CUDA context, or 0 when no context is current or
// the driver does not report one. Host-side caches of per-context state key on it.
unsigned long long current_context_id();

// Program kernel `variant` for `vpt` vectors per thread (1, 2 or 4) on `grid` CTAs of kProgramThreads, or
// in the wide form (vpt 8, where program_variant_has_vpt8) on `grid` CTAs of kProgramWideThreads; the
// schedule `p` by value, or, when `dev` is not null, read from that copy of it in device memory. `order`
// (PdlOrder; other than kPdlWaitFirst with an uploaded schedule only): its place in a batch of independent
// launches; on its own a program waits first and lets the next kernel start at its end.
cudaError_t launch_program(const ProgramParams& p, const ProgramParams* dev, int vpt, int variant, int grid,
                           cudaStream_t s, int order = 0);
// Resident program CTAs per SM (occupancy query; 0 on error).
int program_ctas_per_sm(int vpt, int variant);
cudaError_t device_error_flags_program(unsigned int* flags, bool clear);

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

// Largest grid extent in y and z: rows are laid out over (y, z), so a launch covers up to kMaxGridYZ^2 rows.
constexpr int64_t kMaxGridYZ = 65535;

// Fill a launch configuration: a grid of (ctas_per_row, gy, gz) CTAs with gy * gz >= rows (row index
// y + gy * z, so no CTA divides to find its row; CTAs past the last row return at once), the cluster
// attribute (cluster along x, one row per cluster) when cluster > 1, and PDL.
inline void fill_launch(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, int64_t rows, int ctas_per_row,
                        int threads, int cluster, cudaStream_t s) {
    cfg = cudaLaunchConfig_t{};
    const int64_t gy = rows < kMaxGridYZ ? rows : kMaxGridYZ;
    const int64_t gz = (rows + gy - 1) / gy;
    cfg.gridDim = dim3(static_cast<unsigned>(ctas_per_row), static_cast<unsigned>(gy), static_cast<unsigned>(gz));
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

// Row of this CTA under fill_launch's grid, and its rank (slice) within the row.
__device__ __forceinline__ int64_t launch_row() {
    return static_cast<int64_t>(blockIdx.y) + static_cast<int64_t>(gridDim.y) * blockIdx.z;
}

}  // namespace mbd
