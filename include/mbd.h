/*
 * mbd.h -- C ABI of the memory-bound decoder-layer fusion library (GB300, sm_103a).
 *
 * Four fused, HBM-bound operations of an LLM decoder layer, each one kernel launch on the caller's stream:
 *
 *   mbd_fused_add_rmsnorm            residual <- x + residual; out = RMSNorm(residual) * weight
 *   mbd_fused_add_rmsnorm_quant_fp8  the same, writing FP8 E4M3 codes of the normalised row instead of bf16
 *   mbd_swiglu                       out = silu(gate) * up over a stacked gate_up row
 *   mbd_swiglu_quant_fp8             FP8 E4M3 codes of silu(gate) * up
 *   mbd_fused_add_rmsnorm_quant_nvfp4, mbd_swiglu_quant_nvfp4
 *                                    the norm / SwiGLU with an NVFP4 epilogue (E2M1 codes, E4M3 block scales)
 *   mbd_fused_allreduce_add_rmsnorm[_quant_fp8]
 *                                    the norm fed by n partial activations summed on the way in
 *   mbd_run_program                  a list of the above operations as ONE persistent kernel launch
 *
 * Definitions (cited by page title and section):
 *   [TRT] "TensorRT-LLM: Compiling Inference Engines Ahead of Time", section "Fusing operations, measured":
 *         RMSNorm is the eight-step chain float cast, square, mean, epsilon, reciprocal square root, scaling,
 *         cast to 16 bits and weight multiply; TensorRT-LLM fuses the residual addition into the same kernel
 *         as the normalisation; gate and up come out of one stacked projection and a fused SwiGLU kernel
 *         forms g / (1 + exp(-g)) * up from the two halves.
 *   [FP8] "TensorRT-LLM" architecture walkthrough, "Part V continued: Deep dive: quantization co-designed
 *         with the hardware": FP8 E4M3 is the activation format, with a scale per tensor or per block.
 *   [FP4] same section, NVFP4 paragraph: Blackwell's 4-bit format stores E2M1 elements (sign, 2 exponent bits,
 *         1 mantissa bit, largest magnitude 6); every 16 consecutive elements carry an E4M3 scale and the
 *         tensor an fp32 scale, about 4.5 bits per element in all.
 *   [VLLM] "Introduction to torch.compile and How It Works with vLLM", section 3, custom compiler passes:
 *         a compiler pass replaces SiLU followed by FP8 quantisation with one fused kernel; section 4 reports
 *         a fused AllReduce + RMSNorm + FP8 quantisation as well.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers (or managed memory visible to the device), row-major and
 *     contiguous. bf16 tensors are passed as void* and hold IEEE bfloat16 bit patterns. The caller owns all
 *     memory: the library allocates nothing, never synchronises, keeps no state between calls (apart from
 *     per-device caches of device attributes, kernel attributes and kernel occupancies, keyed by the current
 *     context where they belong to one, and the static schedule buffer's address) and is safe to call from
 *     several host threads.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default stream) and runs in stream
 *     order. Each successful call of an entry point launches exactly one kernel (a batch: one per op).
 *   - Arithmetic is fp32 in registers; every intermediate stays unrounded until the single final rounding
 *     to bf16 or to E4M3 (round to nearest even, saturating finite overflow to +-448).
 *   - Scale convention (both FP8 entry points): `scale` is the DEQUANTISATION multiplier, value ~ code * scale.
 *       MBD_SCALE_STATIC_PER_TENSOR: scale points to ONE fp32 value, read on the device; it must be finite
 *         and > 0 (0 yields all-zero codes; other values give unspecified codes).
 *       MBD_SCALE_DYNAMIC_PER_TOKEN: scale points to n_tokens fp32 values that the kernel WRITES:
 *         scale[t] = amax_t / 448 (fp32) where amax_t is the largest magnitude of row t before quantisation;
 *         a row with amax_t == 0 gets scale 0 and all-zero codes.
 *   - Argument errors are detected on the host before anything is launched; nothing is enqueued then.
 *       MBD_ERR_INVALID_ARG : a null pointer while n_tokens > 0, n_tokens < 0, width <= 0, eps < 0 or not
 *                             finite, an unknown mode, or overlapping buffers other than the allowed alias.
 *       MBD_ERR_MISALIGNED  : a tensor pointer not 16-byte aligned, `scale` not 4-byte aligned, or a width
 *                             not a multiple of 8 elements (one 16-byte vector of bf16).
 *       MBD_ERR_UNSUPPORTED : a shape beyond the limits stated per entry point.
 *       MBD_ERR_CUDA        : the launch itself failed; mbd_last_cuda_error() gives the cudaError_t.
 *     n_tokens == 0 is a no-op returning MBD_OK (pointers are not inspected). Faults during execution
 *     surface at the caller's next synchronisation, as for any kernel.
 */
#ifndef MBD_H
#define MBD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (struct CUstream_st*), declared here so that the header needs no CUDA include. */
typedef struct CUstream_st* mbd_stream_t;

typedef enum {
    MBD_OK = 0,
    MBD_ERR_INVALID_ARG = 1,
    MBD_ERR_MISALIGNED = 2,
    MBD_ERR_UNSUPPORTED = 3,
    MBD_ERR_CUDA = 4
} mbd_status;

typedef enum {
    MBD_SCALE_STATIC_PER_TENSOR = 0,
    MBD_SCALE_DYNAMIC_PER_TOKEN = 1
} mbd_scale_mode;

/* Largest row width (elements) of the entry points that reduce over a row (both norms and
 * mbd_swiglu_quant_fp8 in dynamic mode); wider rows return MBD_ERR_UNSUPPORTED. */
#define MBD_MAX_REDUCED_WIDTH 262144

/* ABI version of this header (bumped on any signature change or added entry point). */
#define MBD_ABI_VERSION 9
int mbd_abi_version(void);

/* Static, human-readable name of a status code (never NULL). */
const char* mbd_status_string(int status);

/* cudaError_t of the most recent MBD_ERR_CUDA returned on the calling host thread (0 if none). */
int mbd_last_cuda_error(void);

/* Number of kernels this library has launched in the process so far (all threads, all devices). */
uint64_t mbd_kernel_launches(void);

/* Device-side error bits. A kernel that splits a row over a thread-block cluster exchanges partial sums
 * through distributed shared memory and waits for its peers with a bounded wait (about one second); if
 * the wait ever ran out, the kernel set this bit and returned without writing its outputs. */
#define MBD_DEVERR_EXCHANGE_TIMEOUT 1u

/* Copy the OR of the library's device error words on the CURRENT device into *flags and, if clear != 0,
 * reset them. Synchronous (a device-to-host copy on the legacy default stream). Returns MBD_ERR_INVALID_ARG
 * for a null flags pointer, MBD_ERR_CUDA if the copy fails. */
mbd_status mbd_device_error_flags(uint32_t* flags, int clear);

/* Self-test of the failure path (no counterpart on the source pages): launches one warp that waits on an
 * mbarrier which nothing will ever complete, with a wait limit of limit_cycles SM clock cycles
 * (1 <= limit_cycles <= 2^31, about one second at 2 GHz). The wait runs out, the kernel sets
 * MBD_DEVERR_EXCHANGE_TIMEOUT and returns; the context stays usable. Returns MBD_ERR_INVALID_ARG for a
 * limit out of range. Asynchronous on `stream` like every launch. */
mbd_status mbd_selftest_bounded_wait(uint64_t limit_cycles, mbd_stream_t stream);

/*
 * Fused residual add + RMSNorm [TRT].
 *   For every row t < n_tokens and column j < hidden:
 *     s[t,j]        = bf16(x[t,j] + residual[t,j])            (fp32 add, one rounding)
 *     residual[t,j] = s[t,j]                                  (written back in place)
 *     inv_t         = 1 / sqrt(sum_j s[t,j]^2 / hidden + eps)
 *     out[t,j]      = bf16(weight[j] * s[t,j] * inv_t)
 *   out      : [n_tokens, hidden] bf16, written. May be the same pointer as x (in-place); must not
 *              overlap residual or weight otherwise.
 *   residual : [n_tokens, hidden] bf16, read and overwritten with s.
 *   x        : [n_tokens, hidden] bf16, read.
 *   weight   : [hidden] bf16, read.
 *   eps      : >= 0, added to the mean of squares inside the square root.
 *   Limits   : hidden <= MBD_MAX_REDUCED_WIDTH.
 */
mbd_status mbd_fused_add_rmsnorm(void* out, void* residual, const void* x, const void* weight,
                                 int64_t n_tokens, int64_t hidden, float eps, mbd_stream_t stream);

/*
 * Fused residual add + RMSNorm + FP8 E4M3 quantisation [TRT], [FP8], [VLLM] (the norm-and-quantise half
 * of AllReduce + RMSNorm + Quant, on one GPU).
 *   s, residual and inv_t as in mbd_fused_add_rmsnorm; v[t,j] = weight[j] * s[t,j] * inv_t in fp32 (not
 *   rounded to bf16), and out_q[t,j] = e4m3(v[t,j] / scale) with the scale of the row (see conventions).
 *   out_q    : [n_tokens, hidden] uint8 E4M3 codes, written; must not overlap any other argument.
 *   scale    : static -> [1] fp32 read; dynamic -> [n_tokens] fp32 written (must not overlap others).
 *   Only the codes are written, not the bf16 normalised row.
 *   Limits   : hidden <= MBD_MAX_REDUCED_WIDTH.
 */
mbd_status mbd_fused_add_rmsnorm_quant_fp8(uint8_t* out_q, void* residual, const void* x,
                                           const void* weight, int64_t n_tokens, int64_t hidden, float eps,
                                           mbd_scale_mode mode, float* scale, mbd_stream_t stream);

/* Largest number of partial activations of the all-reduce entry points below. */
#define MBD_MAX_PARTIALS 8

/*
 * The single-GPU half of AllReduce + RMSNorm [VLLM] section 4 (fused AllReduce + RMSNorm, with or without
 * FP8 quantisation): n_partials partial activations -- one per tensor-parallel rank, already gathered on
 * this GPU -- are reduced and fed to the fused residual add + RMSNorm, in one pass:
 *     x[t,j] = bf16(sum_k partials[k][t,j])   (the exact sum rounded once: what a bf16 all-reduce delivers)
 * then everything as in mbd_fused_add_rmsnorm (bf16 out) / mbd_fused_add_rmsnorm_quant_fp8 (E4M3 codes).
 * With n_partials == 1 the results are bit-identical to those entry points.
 *   partials   : HOST array of n_partials DEVICE pointers, each [n_tokens, hidden] bf16, 16-byte aligned,
 *                read only; 1 <= n_partials <= MBD_MAX_PARTIALS. They may repeat or overlap each other but
 *                not residual, weight, out (bf16 out may be exactly partials[0]) or a dynamic scale.
 *   other arguments and errors: as for the plain entry points. Limit: hidden <= 32768 (one 8-element vector
 *   of exact partial sums per thread, at most 8 CTAs of 512 threads per row); wider rows return
 *   MBD_ERR_UNSUPPORTED.
 */
mbd_status mbd_fused_allreduce_add_rmsnorm(void* out, void* residual, const void* const* partials, int n_partials,
                                           const void* weight, int64_t n_tokens, int64_t hidden, float eps,
                                           mbd_stream_t stream);
mbd_status mbd_fused_allreduce_add_rmsnorm_quant_fp8(uint8_t* out_q, void* residual, const void* const* partials,
                                                     int n_partials, const void* weight, int64_t n_tokens,
                                                     int64_t hidden, float eps, mbd_scale_mode mode, float* scale,
                                                     mbd_stream_t stream);

/*
 * SwiGLU over the stacked gate_up projection [TRT].
 *   gate_up : [n_tokens, 2 * inter] bf16, read; columns 0..inter-1 are gate, inter..2*inter-1 are up.
 *   out     : [n_tokens, inter] bf16, written: out[t,j] = bf16(silu(g) * u), silu(g) = g / (1 + exp(-g)),
 *             computed in fp32 without rounding silu(g) first. Must not overlap gate_up.
 */
mbd_status mbd_swiglu(void* out, const void* gate_up, int64_t n_tokens, int64_t inter, mbd_stream_t stream);

/*
 * Quantize(SiLU(gate) * up) [VLLM], [FP8].
 *   h[t,j] = silu(g) * u in fp32 (as mbd_swiglu, not rounded to bf16); out_q[t,j] = e4m3(h[t,j] / scale).
 *   out_q   : [n_tokens, inter] uint8 E4M3 codes, written; must not overlap gate_up or scale.
 *   scale   : static -> [1] fp32 read; dynamic -> [n_tokens] fp32 written.
 *   Limits  : dynamic mode needs inter <= MBD_MAX_REDUCED_WIDTH.
 */
mbd_status mbd_swiglu_quant_fp8(uint8_t* out_q, const void* gate_up, int64_t n_tokens, int64_t inter,
                                mbd_scale_mode mode, float* scale, mbd_stream_t stream);

/*
 * NVFP4 epilogues [FP4] of the fused residual add + RMSNorm and of SwiGLU. The row values v (the norm's
 * v[t,j] = weight[j] * s[t,j] * inv_t, SwiGLU's h[t,j], both fp32, not rounded) are cut into blocks of 16
 * consecutive elements; with S = *tensor_scale and amax_b the largest |v| of block b:
 *     out_sf[t,b]  = e4m3(amax_b / (6 S))                    block scale, so that amax_b maps to about 6
 *     code[t,j]    = e2m1(v[t,j] / (dec(out_sf[t,b]) S))     0 where the block scale is 0
 * e2m1 rounds to nearest even among 0, 0.5, 1, 1.5, 2, 3, 4, 6, saturates at 6 and keeps the sign (also on
 * a zero); the value is v ~ dec(code) * dec(out_sf) * S. The fp32 arithmetic (the divisions by 6 S and S
 * folded into per-row constants, 1 / dec(out_sf) from the hardware reciprocal) sits within a few ulps of
 * the exact ratios, so a value within that distance of a rounding midpoint may round the other way.
 *   out_q        : [n_tokens, width / 2] uint8, written: element 2i in the low nibble of byte i, 2i + 1 in
 *                  the high nibble, bit 3 of a nibble the sign. 16-byte aligned.
 *   out_sf       : [n_tokens, width / 16] uint8 E4M3 block scales, written, row-major (no tensor-core
 *                  swizzle). Any alignment.
 *   tensor_scale : ONE fp32 value S, read on the device, 4-byte aligned; usable range 2^-64 <= S <= 2^64.
 *                  Anything else (0, negative, NaN, infinite, or outside that range) gives all-zero block
 *                  scales and codes.
 *   Other arguments as in mbd_fused_add_rmsnorm / mbd_swiglu. out_q, out_sf and tensor_scale must not
 *   overlap anything written; tensor_scale may overlap inputs. width (hidden or inter) must be a multiple of
 *   16 elements, else MBD_ERR_MISALIGNED; the norm's limit is hidden <= MBD_MAX_REDUCED_WIDTH.
 */
mbd_status mbd_fused_add_rmsnorm_quant_nvfp4(uint8_t* out_q, uint8_t* out_sf, void* residual, const void* x,
                                             const void* weight, int64_t n_tokens, int64_t hidden, float eps,
                                             const float* tensor_scale, mbd_stream_t stream);
mbd_status mbd_swiglu_quant_nvfp4(uint8_t* out_q, uint8_t* out_sf, const void* gate_up, int64_t n_tokens,
                                  int64_t inter, const float* tensor_scale, mbd_stream_t stream);

/*
 * Programs: several operations in one persistent kernel launch. No counterpart on the source pages as an
 * API; it is this library's form of the launch-overhead remedies they discuss: [TRT] "Fusing operations,
 * measured" notes that on a data-center GPU issuing the kernels can take longer than running them, and
 * "Leaving the engine behind" lists CUDA graphs captured per batch size for decoding; [VLLM] section 5
 * plans a single kernel for a whole forward pass.
 *
 * Each op is one call of the entry points above, described by value. Every op's n_tokens rows are
 * independent: row t of an op reads and writes only row t of its tensors (plus the shared weight and a
 * static scale). The program therefore gives the results of calling the ops one after another on
 * `stream`, provided every buffer that two ops share, with one of them writing it, is the SAME tensor in
 * both: the same pointer and the same row layout (same n_tokens and bytes per row) -- typically the
 * residual that consecutive norms update, or an output that a later op reads in place. Ops linked that way
 * form a chain whose rows run op after op inside one CTA; ops that share nothing with another op are spread
 * over all CTAs. Sharing that is not row-aligned (a different pointer into the same memory, a different
 * row layout, a dynamic scale read as a static scale) returns MBD_ERR_UNSUPPORTED.
 */
typedef enum {
    MBD_OP_ADD_RMSNORM = 0,              /* mbd_fused_add_rmsnorm: in = x, out bf16 */
    MBD_OP_ADD_RMSNORM_QUANT_FP8 = 1,    /* mbd_fused_add_rmsnorm_quant_fp8: mode, scale */
    MBD_OP_ADD_RMSNORM_QUANT_NVFP4 = 2,  /* mbd_fused_add_rmsnorm_quant_nvfp4: out_sf, scale = tensor scale */
    MBD_OP_SWIGLU = 3,                   /* mbd_swiglu: in = gate_up */
    MBD_OP_SWIGLU_QUANT_FP8 = 4,         /* mbd_swiglu_quant_fp8: mode, scale */
    MBD_OP_SWIGLU_QUANT_NVFP4 = 5        /* mbd_swiglu_quant_nvfp4: out_sf, scale = tensor scale */
} mbd_op_kind;

/* One operation of a program: the arguments of its entry point (unused fields are ignored). */
typedef struct {
    int32_t kind;           /* mbd_op_kind */
    int32_t mode;           /* FP8 ops: mbd_scale_mode */
    int64_t n_tokens;
    int64_t width;          /* hidden (norms) or inter (SwiGLU) */
    float eps;              /* norms */
    int32_t reserved;       /* must be 0 */
    void* out;              /* bf16, E4M3 codes or packed E2M1 codes */
    uint8_t* out_sf;        /* NVFP4 block scales */
    void* residual;         /* norms */
    const void* in;         /* norms: x; SwiGLU: gate_up */
    const void* weight;     /* norms */
    float* scale;           /* FP8 scale ([1] read or [n_tokens] written), or the NVFP4 tensor scale ([1] read) */
} mbd_op;

/* Largest number of ops in one program. */
#define MBD_MAX_PROGRAM_OPS 128
/* Largest hidden size of a norm in a program: one CTA of 256 threads holds the row, 4 vectors per thread.
 * SwiGLU rows of any width run in chunks. A dynamic FP8 SwiGLU row of up to 16384 elements is held whole by
 * one CTA (1024 threads, 2 vectors each) in the programs whose epilogue sets include it, except where the
 * program's chained norms run at one vector per thread (rows of up to 2048 elements), which keeps 256-thread
 * CTAs; a row wider than its CTA holds takes two passes: the row maximum, then the codes from the same
 * inputs, read again from L2. */
#define MBD_MAX_PROGRAM_WIDTH 8192

/*
 * Run ops[0..n_ops) as one persistent kernel on `stream`.
 *   ops    : HOST array of n_ops descriptors, read during the call only (the schedule travels in the kernel's
 *            parameters; nothing is allocated or copied beforehand).
 *   n_ops  : 0 (no-op) .. MBD_MAX_PROGRAM_OPS.
 * Each op is validated exactly as its entry point validates it (and the same status is returned, nothing
 * launched). Besides: an unknown kind or a non-zero `reserved` gives MBD_ERR_INVALID_ARG; a norm wider
 * than MBD_MAX_PROGRAM_WIDTH, sharing that is not row-aligned, or epilogues outside the compiled sets
 * gives MBD_ERR_UNSUPPORTED. The compiled sets (norm epilogues / SwiGLU epilogues), of which a program
 * takes the first that covers its ops: bf16 / bf16; FP8 static / FP8 dynamic; NVFP4 / NVFP4; bf16 and FP8
 * static / bf16, FP8 static and FP8 dynamic (bf16 and FP8 ops mixed in one launch). A dynamic-FP8 norm
 * therefore runs only in the single-call entry points. Ops with n_tokens == 0 are skipped; if nothing
 * remains, nothing is launched.
 * Reductions run inside one CTA per row (no cluster), so sums may round differently from the single-call
 * entry points in their last bit, and consecutive norms on one residual row form 1/sqrt(mean + eps) with the
 * hardware reciprocal square root (a few ulps); every result keeps the tolerances stated for those entry
 * points.
 */
mbd_status mbd_run_program(const mbd_op* ops, int n_ops, mbd_stream_t stream);

/*
 * A batch of independent ops, each run by its own single-call kernel with the launch shape its entry point
 * would use, the launches overlapping one another. No counterpart on the source pages as an API; it answers
 * [TRT] "Fusing operations, measured" on the cost of many short launches for batches too large for a
 * program: a call of about a thousand rows streams its bytes in a few microseconds, about as long as a
 * launch takes to ramp up and drain, and here each launch after the first starts while the one before it
 * still runs.
 *   ops    : HOST array of n_ops descriptors (mbd_op, as in programs), read during the call only.
 *   n_ops  : 0 (no-op) .. MBD_MAX_INDEPENDENT_OPS.
 * The ops must be independent: no op may read or write memory that another op of the batch writes (its
 * output, residual, block scales or dynamic scales); sharing read-only memory (a weight, a static scale) is
 * allowed. Results are bit-identical to calling the entry points one after another on `stream`, in any
 * order. Stream order holds for the batch as a whole: the first launch waits for the work enqueued before
 * the call, and work enqueued after the call starts only once every op of the batch has completed.
 * Each op is validated exactly as its entry point validates it (same status, nothing launched); besides,
 * an unknown kind or a non-zero `reserved` gives MBD_ERR_INVALID_ARG, and so does a pair of ops that are not
 * independent. All checks run before the first launch; a launch failure returns MBD_ERR_CUDA with the ops
 * before it enqueued. Ops with n_tokens == 0 are skipped. One launch per remaining op.
 */
#define MBD_MAX_INDEPENDENT_OPS 64
mbd_status mbd_run_independent(const mbd_op* ops, int n_ops, mbd_stream_t stream);


/*
 * The same in two steps, for a program that runs many times (every decode step): build validates and
 * schedules once on the host; launch enqueues the kernel with no further host work beyond the launch
 * itself. mbd_run_program is build + launch, and checking and scheduling ~100 ops costs tens of
 * microseconds of host time per call.
 *   mbd_program_plan : plain caller-owned memory (may be copied, stored or freed; holds no pointer into
 *                      itself), filled by build. It records the device that was current at build time
 *                      (launch shapes depend on its SM count) and the ops' device pointers: the tensors must
 *                      stay where they are while the plan is launched.
 *   build  : the checks and statuses of mbd_run_program; on failure the plan is left unusable. No kernel
 *            is launched (device attributes are queried).
 *   launch : MBD_ERR_INVALID_ARG for a plan that build did not fill, or on a device other than the one it
 *            was built on; a plan with nothing to do launches nothing and returns MBD_OK.
 */
#define MBD_PROGRAM_PLAN_BYTES 16384
typedef struct {
    uint64_t opaque[MBD_PROGRAM_PLAN_BYTES / 8];
} mbd_program_plan;

mbd_status mbd_program_plan_build(const mbd_op* ops, int n_ops, mbd_program_plan* plan);
mbd_status mbd_program_plan_launch(const mbd_program_plan* plan, mbd_stream_t stream);

/*
 * A plan's schedule kept in device memory. mbd_program_plan_launch passes the whole schedule (about 14 KB)
 * in the kernel parameters, and such a launch costs tens of microseconds of host time; after one upload,
 * launch_uploaded passes a single pointer.
 *   mbd_program_schedule_bytes : device bytes a schedule takes (a multiple of 256).
 *   upload  : one asynchronous host-to-device copy of the plan's schedule into `schedule` (caller-owned
 *             device memory, 256-byte aligned, at least mbd_program_schedule_bytes() long) on `stream`.
 *             The plan must stay unchanged until the copy has executed (it may read the plan after the
 *             call returns). MBD_ERR_INVALID_ARG: an unfilled plan, a null or short buffer;
 *             MBD_ERR_MISALIGNED: a buffer not 256-byte aligned; MBD_ERR_CUDA: the copy failed.
 *   launch_uploaded : the kernel reads the schedule from `schedule`, which must hold this plan's upload
 *             (stream order makes an upload on the same stream visible to the launch). Errors as for
 *             mbd_program_plan_launch, plus those of the buffer. `schedule` must not be written while the
 *             kernel runs.
 */
size_t mbd_program_schedule_bytes(void);
mbd_status mbd_program_plan_upload(const mbd_program_plan* plan, void* schedule, size_t schedule_bytes,
                                   mbd_stream_t stream);
mbd_status mbd_program_plan_launch_uploaded(const mbd_program_plan* plan, const void* schedule, mbd_stream_t stream);

/*
 * A batch of independent ops (mbd_run_independent) with a program in front of it: the program (`plan` with its schedule uploaded to `schedule`,
 * as for mbd_program_plan_launch_uploaded) launches first and lets the ops' launches start once the work
 * before the call is complete, so small, latency-bound rows (the program) run beside large, bandwidth-bound
 * ones (the ops). No op may read or write memory that the program writes, nor the reverse (checked for every
 * pair of a program op and a batch op, so the host checks grow with their product); within the program the
 * program's own rules apply. Stream order holds for the whole: the program waits for the work enqueued
 * before the call, and work enqueued after it starts once the program and every op have completed. Results
 * are bit-identical to launching the program, then calling the ops, one after another.
 * Errors: those of mbd_program_plan_launch_uploaded (a null, unfilled or other-device plan, a null or
 * misaligned schedule) and of mbd_run_independent; MBD_ERR_INVALID_ARG also when an op and the program are not
 * independent. A plan with nothing to do launches only the ops, as mbd_run_independent does.
 */
mbd_status mbd_run_independent_with_program(const mbd_program_plan* plan, const void* schedule, const mbd_op* ops,
                                            int n_ops, mbd_stream_t stream);

/*
 * mbd_program_plan_upload + mbd_program_plan_launch_uploaded without caller memory. No counterpart on the
 * source pages: it exists for callers that cannot allocate device memory. Examples are serving engines that
 * reserve nearly all of HBM for their own pool (KV cache, weights) and hand kernels only the tensors they
 * own, plug-in interfaces that pass a kernel its inputs and outputs and nothing else, and latency-critical
 * loops where cudaMalloc (which may synchronise the device) is not acceptable.
 * The schedule is copied (one asynchronous host-to-device copy on `stream`, as upload does) into a static
 * buffer of the library: MBD_STATIC_SCHEDULE_BYTES per device, part of the library's device image and held
 * by every GPU that loads the library until the process exits. The first call on a device looks up the
 * buffer's device address (cudaGetSymbolAddress, with that device current) and caches it together with the
 * id of the current CUDA context; a call made in another context of that device (for instance after
 * cudaDeviceReset has re-created the primary context, whose module image may sit elsewhere) looks it up
 * again. Make the first call on a device, and the first after a reset, before any stream capture. Nothing is
 * allocated (no cudaMalloc, cudaFree or other allocating call). Every call overwrites the buffer's whole
 * schedule record with its own plan's, so plans may alternate freely; because the buffer is shared, calls
 * that overlap on the GPU race (e.g. on different streams of one device) and must not be issued; calls on
 * one stream are ordered. Every schedule the build accepts fits the buffer (a compile-time check of the
 * library), so no plan is refused for its size. Errors as for mbd_program_plan_launch; MBD_ERR_CUDA also
 * when the current device cannot be read or the address lookup fails (mbd_last_cuda_error has the cause).
 */
#define MBD_STATIC_SCHEDULE_BYTES 16384
mbd_status mbd_program_plan_launch_static(const mbd_program_plan* plan, mbd_stream_t stream);

/*
 * Launch-shape tuning (shape-bucket dispatch). [TRT] "Auto-tuning, measured": TensorRT-LLM picks kernel
 * tactics per shape bucket at startup and keeps them in a cache that can be saved to a file and reloaded.
 * Here the knobs are the launch shape of the single-call entry points: CTAs per row (one thread-block
 * cluster when the row is reduced), 16-byte vectors per thread and threads per CTA. Without a table the
 * built-in rules choose (they come from sweeps on GB300). A table is a list of entries; a call takes the
 * FIRST entry whose kind (and FP8 mode) matches and whose token and width buckets hold it, provided its
 * shape fits the call (enough threads x vectors for a slice of the row, at most 8 CTAs when the row is
 * reduced); otherwise the next matching entry, then the rules. The all-reduce and program entry points do
 * not use the table. One shape is fixed by the rules alone: a dynamic-FP8 SwiGLU of at least 4 rows per SM
 * with rows of 4609 to 10240 vectors (inter 36872 to 81920) brings its row slices into shared memory by
 * bulk copies (clusters of 7, or 8 past 8960 vectors, 4 vectors per thread), whatever the table says. The
 * tuner that fills it is memory_bound_decoder_gb300/tune.py.
 */
typedef struct {
    int32_t kind;                 /* mbd_op_kind of the entry point */
    int32_t mode;                 /* FP8 kinds: mbd_scale_mode; ignored otherwise */
    int64_t tokens_min, tokens_max;  /* n_tokens bucket, inclusive */
    int64_t width_min, width_max;    /* hidden / inter bucket, inclusive */
    int32_t ctas_per_row;         /* >= 1 */
    int32_t vectors_per_thread;   /* 1, 2, 4 or 8 */
    int32_t threads;              /* 32 .. 512, a multiple of 32 */
    int32_t reserved;             /* 0 */
} mbd_tuning_entry;

#define MBD_MAX_TUNING_ENTRIES 4096

/* Replace the process-wide table with a copy of entries[0 .. n_entries) (n_entries == 0: no table, the rules
 * alone). Thread-safe: a call in flight on another thread uses either the old or the new table. Returns
 * MBD_ERR_INVALID_ARG (table unchanged) for a bad count, null entries, or an entry with an unknown kind or
 * FP8 mode, an empty bucket, a non-zero reserved field or a shape outside the ranges above. */
mbd_status mbd_tuning_set(const mbd_tuning_entry* entries, int n_entries);

/* The number of entries in the table; copies the first min(that, capacity) into entries (may be NULL). */
int mbd_tuning_get(mbd_tuning_entry* entries, int capacity);

/* The launch shape (CTAs per row after rounding, vectors per thread, threads) that a call of entry point
 * `kind` (FP8: with `mode`) on n_tokens x width would use now (table, else rules), without launching. Uses
 * the current device's SM count. Errors: MBD_ERR_INVALID_ARG (unknown kind or mode, n_tokens or width <= 0,
 * a null output), the width checks of the entry point (MBD_ERR_MISALIGNED, MBD_ERR_UNSUPPORTED). */
mbd_status mbd_launch_shape(int kind, int mode, int64_t n_tokens, int64_t width, int32_t* ctas_per_row,
                            int32_t* vectors_per_thread, int32_t* threads);

#ifdef __cplusplus
}
#endif

#endif /* MBD_H */
