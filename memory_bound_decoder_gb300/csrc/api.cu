// C ABI of the fusion library: host-side argument checks, launch-shape selection and dispatch.
// Every check runs before anything is enqueued; a failing call launches nothing.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstddef>
#include <cstdint>
#include <memory>
#include <vector>

#include <cuda.h>

#include "mbd.h"
#include "launch.h"

namespace mbd {

unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    struct Entry {
        GetCurrent get_current = nullptr;
        GetId get_id = nullptr;
    };
    // Driver entry points through the runtime, so the library links no driver library at build time.
    static const Entry entry = [] {
        Entry f;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_current = reinterpret_cast<GetCurrent>(p);
        p = nullptr;
        q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_id = reinterpret_cast<GetId>(p);
        (void)cudaGetLastError();
        return f;
    }();
    if (!entry.get_current || !entry.get_id) return 0;
    CUcontext ctx = nullptr;
    if (entry.get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    if (entry.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

}  // namespace mbd

namespace {

thread_local int g_last_cuda_error = 0;
std::atomic<uint64_t> g_launches{0};

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];  // 0 = not queried yet

int sm_count_of_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        return 148;
    }
    g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Half-open byte ranges [a, a + na) and [b, b + nb) intersect.
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return na > 0 && nb > 0 && x < y + nb && y < x + na;
}

constexpr int kMaxClusterCtas = 8;   // portable cluster size (also the exchange's slot count)
constexpr int kMaxThreads = 512;     // matches __launch_bounds__ of the kernels

// What a launch reduces over each row: the norm's sum of squares, the dynamic SwiGLU's max |h|, or
// nothing (pure streams, whose row slices are independent CTAs without a cluster).
enum class Shape { kNorm, kNormPartials, kRowMax, kStream };

int cdiv(int a, int b) { return (a + b - 1) / b; }

// Launch shape, chosen from a sweep of CTAs per row x vectors per thread x threads on GB300 (back-to-back
// launches; inputs larger than L2 for the large batches):
//  - at least one row per SM (large batches):
//      norm: one CTA per row while the row fits 512 threads x 4 vectors (hidden <= 16384), 4 vectors per
//            thread from 512 vectors per row up (the tuner: +6 to +22% at hidden 4096 to 8192 over 2 per
//            thread), else the fewest (>= 2) that keep the CTA at <= 512 threads -- no cluster exchange;
//      dynamic SwiGLU: rows cut into slices of about 576 vectors over a cluster of at most 8 CTAs,
//            2 vectors per thread (with the wave-ahead L2 warming, 8 x 416 threads beat 7 x 480 by 4 to
//            6% at I 53248 and 1024 to 4096 tokens; at one to four rows per SM, where no warming runs,
//            clusters of 7 stay ahead);
//      streams: slices of <= 1024 vectors, <= 256 threads;
//      NVFP4 (more work per vector): the norm takes 4 vectors per thread (34.6 vs 43.0 us at T 4096,
//            H 8192), the SwiGLU stream ~448-vector slices at 2 vectors per thread (76.8 vs 81.5 us at
//            T 2048, I 53248; 80.7 vs 87.3 us at T 4096, I 28672);
//      norm over partial activations: one vector per thread, ~256-vector slices over up to 8 CTAs (the
//            slices of the partials come into shared memory by bulk copies).
//  - one to four rows per SM: the norm stays in one CTA with the fewest vectors per thread that fit 512
//    threads (a cluster exchange costs +50% there), the bf16 and FP8 streams take ~256-vector slices (the
//    tuner: +26 to +57% over the large-batch shapes at 256 tokens);
//  - fewer rows than SMs (decode): latency-bound. Norm rows are cut into slices of about 256 vectors, the
//    dynamic SwiGLU's into up to 8 slices of up to 512 threads at one vector each (the tuner: +12 to +49%
//    at 4 to 64 tokens); bf16 and FP8 streams are split until about six CTAs per SM pull bytes at once,
//    in slices of at least 64 vectors (+30 to +95% at 64 tokens over two CTAs per SM), NVFP4 streams until
//    about two. At most 256 threads per CTA except the dynamic SwiGLU.
// `pairs` (NVFP4): slices of an even number of vectors, so that every 16-element block lies in one CTA, in
// neighbouring lanes.
bool plan_rows(int64_t rows, int nvec, Shape shape, int sms, bool pairs, mbd::RowPlan* plan) {
    *plan = mbd::RowPlan{};
    const bool reduces = shape != Shape::kStream;
    const bool small = rows < sms;
    const bool mid = !small && rows < 4 * int64_t{sms};   // one to four rows per SM
    int c;
    int min_vpt = (shape == Shape::kStream || small) ? 1 : 2;
    int max_threads = (shape == Shape::kStream || small) ? 256 : kMaxThreads;
    if (shape == Shape::kNorm) {
        if (small) {
            c = cdiv(nvec, 256);
        } else if (mid) {        // one CTA per row (no cluster), the fewest vectors per thread for <= 512 threads
            c = cdiv(nvec, 2048);
            min_vpt = 1;
        } else {
            c = cdiv(nvec, 2048);
            if (pairs || nvec >= 512) min_vpt = 4;
        }
    } else if (shape == Shape::kNormPartials) {   // one vector per thread (the partials' slices in shared memory)
        c = cdiv(nvec, 256);   // slices of ~256 vectors (8 x 256 threads at H 16384): at H 5120 and 8192 they
                               // beat ~128 by 8 to 26%, at H 16384 rows over 4 x 512 lose 3%
    } else if (shape == Shape::kRowMax) {
        if (small) {             // up to 8 CTAs of up to 512 threads, one vector each where the row allows
            c = cdiv(nvec, 256);
            if (c > 8) c = 8;
            max_threads = kMaxThreads;
        } else {                 // clusters of up to 7 CTAs, 8 where the wave-ahead warming runs (below)
            c = cdiv(nvec, 576);
            const int cap = mid ? 7 : 8;
            if (c > cap) c = cap;
        }
    } else if (pairs) {
        c = cdiv(nvec, 448);
        if (small) {
            int want = static_cast<int>((2 * sms + rows - 1) / rows);  // about two CTAs per SM
            const int by_width = cdiv(nvec, 32);                        // at least a warp of vectors per CTA
            if (want > by_width) want = by_width;
            if (want > c) c = want;
        } else {
            min_vpt = 2;
        }
    } else {
        c = cdiv(nvec, mid ? 256 : 1024);
        if (small) {
            int want = static_cast<int>((6 * sms + rows - 1) / rows);  // about six CTAs per SM
            const int by_width = cdiv(nvec, 64);                        // slices of at least 64 vectors
            if (want > by_width) want = by_width;
            if (want > c) c = want;
        }
    }
    const int widest = (shape == Shape::kNormPartials ? 1 : 8) * kMaxThreads;  // vectors one CTA can take
    if (c < cdiv(nvec, widest)) c = cdiv(nvec, widest);
    if (reduces && c > kMaxClusterCtas) c = kMaxClusterCtas;
    if (c < 1) c = 1;
    int slice = cdiv(nvec, c);
    if (pairs && (slice & 1)) ++slice;
    c = cdiv(nvec, slice);  // no empty slice
    const int max_vpt = shape == Shape::kNormPartials ? 1 : 8;
    int vpt = 0;
    for (int v : {1, 2, 4, 8}) {
        if (v >= min_vpt && v <= max_vpt && cdiv(slice, v) <= max_threads) {
            vpt = v;
            break;
        }
    }
    if (vpt == 0) vpt = max_vpt;  // very wide rows: as many threads as needed
    const int threads = cdiv(cdiv(slice, vpt), 32) * 32;
    if (threads > kMaxThreads) return false;
    plan->ctas_per_row = c;
    plan->slice = slice;
    plan->threads = threads;
    plan->vpt = vpt;
    plan->prefetch = small ? 1 : 0;
    // Large dynamic-SwiGLU launches: warm L2 half a wave ahead (the rows resident at once: SMs x CTAs per SM,
    // by threads at the <= 32 registers of 1-2 vectors per thread, over the CTAs per row), one bulk prefetch
    // per slice: 87.1 vs 99.6 us without at T 2048, I 53248 (8 x 416 threads; 91.6 with per-vector
    // prefetches), 84.7 vs 92.6 at T 4096, I 28672; a quarter or twice the distance is no better. No gain
    // for the norms.
    if (shape == Shape::kRowMax && !small && !mid && vpt <= 2)
        plan->ahead = static_cast<int>(int64_t{sms} * (2048 / threads) / c / 2);
    return rows <= mbd::kMaxGridYZ * mbd::kMaxGridYZ;
}

mbd_status finish_launch(cudaError_t e) {
    if (e != cudaSuccess) {
        g_last_cuda_error = static_cast<int>(e);
        (void)cudaGetLastError();
        return MBD_ERR_CUDA;
    }
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return MBD_OK;
}

mbd_status check_width(int64_t n_tokens, int64_t width) {
    if (n_tokens < 0 || width <= 0) return MBD_ERR_INVALID_ARG;
    if (width % 8 != 0) return MBD_ERR_MISALIGNED;
    if (width > (int64_t{1} << 28)) return MBD_ERR_UNSUPPORTED;
    return MBD_OK;
}

// Output bytes of T x width elements under an epilogue: bf16 2, E4M3 1, packed E2M1 1/2 per element.
size_t out_bytes(mbd::Epilogue ep, int64_t n_tokens, int64_t width) {
    const size_t n = static_cast<size_t>(n_tokens) * static_cast<size_t>(width);
    return ep == mbd::kBf16 ? 2 * n : (ep == mbd::kNvfp4 ? n / 2 : n);
}

// The FP8 epilogue of a scale mode, false for an unknown mode.
bool fp8_epilogue(int mode, mbd::Epilogue* ep) {
    if (mode == MBD_SCALE_STATIC_PER_TENSOR) *ep = mbd::kFp8Static;
    else if (mode == MBD_SCALE_DYNAMIC_PER_TOKEN) *ep = mbd::kFp8Dynamic;
    else return false;
    return true;
}

// Every host-side check of one norm call, then its kernel parameters in *p (p->rows == 0: nothing to do).
mbd_status norm_prepare(void* out, uint8_t* out_sf, mbd::Epilogue ep, void* residual, const void* x,
                        const void* weight, int64_t n_tokens, int64_t hidden, float eps, float* scale,
                        const void* const* partials, int n_partials, mbd::NormParams* p) {
    *p = mbd::NormParams{};
    mbd_status st = check_width(n_tokens, hidden);
    if (st != MBD_OK) return st;
    const bool quant = ep != mbd::kBf16, dyn = ep == mbd::kFp8Dynamic, fp4 = ep == mbd::kNvfp4;
    if (fp4 && hidden % 16 != 0) return MBD_ERR_MISALIGNED;
    if (!(eps >= 0.0f) || !std::isfinite(eps)) return MBD_ERR_INVALID_ARG;
    if (hidden > MBD_MAX_REDUCED_WIDTH) return MBD_ERR_UNSUPPORTED;
    if (partials && (n_partials < 1 || n_partials > MBD_MAX_PARTIALS)) return MBD_ERR_INVALID_ARG;
    if (n_tokens == 0) return MBD_OK;
    if (partials) x = partials[0];   // validated below like x; the others are checked in the loop
    if (!out || !residual || !x || !weight || (quant && !scale) || (fp4 && !out_sf)) return MBD_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(residual, 16) || !aligned(x, 16) || !aligned(weight, 16) ||
        (quant && !aligned(scale, 4)))
        return MBD_ERR_MISALIGNED;
    const size_t act = static_cast<size_t>(n_tokens) * static_cast<size_t>(hidden) * 2;
    const size_t outb = out_bytes(ep, n_tokens, hidden);
    const size_t sfb = fp4 ? static_cast<size_t>(n_tokens) * static_cast<size_t>(hidden / 16) : 0;
    const size_t wb = static_cast<size_t>(hidden) * 2;
    const size_t sb = quant ? (dyn ? static_cast<size_t>(n_tokens) * 4 : 4) : 0;
    if (overlap(residual, act, x, act) || overlap(residual, act, weight, wb)) return MBD_ERR_INVALID_ARG;
    if (overlap(out, outb, residual, act) || overlap(out, outb, weight, wb)) return MBD_ERR_INVALID_ARG;
    // out may alias x exactly (bf16 only); any other overlap with x is rejected
    if (overlap(out, outb, x, act) && !(!quant && out == x)) return MBD_ERR_INVALID_ARG;
    if (fp4 && (overlap(out_sf, sfb, out, outb) || overlap(out_sf, sfb, residual, act) ||
                overlap(out_sf, sfb, x, act) || overlap(out_sf, sfb, weight, wb) || overlap(out_sf, sfb, scale, sb)))
        return MBD_ERR_INVALID_ARG;
    if (dyn && (overlap(scale, sb, out, outb) || overlap(scale, sb, residual, act) ||
                overlap(scale, sb, x, act) || overlap(scale, sb, weight, wb)))
        return MBD_ERR_INVALID_ARG;
    // a read-only scale (FP8 static, NVFP4) may share memory with the inputs but not with what is written
    if (quant && !dyn && (overlap(scale, sb, out, outb) || overlap(scale, sb, residual, act)))
        return MBD_ERR_INVALID_ARG;
    for (int k = 1; partials && k < n_partials; ++k) {   // partial 0 was checked as x above
        const void* pk = partials[k];
        if (!pk) return MBD_ERR_INVALID_ARG;
        if (!aligned(pk, 16)) return MBD_ERR_MISALIGNED;
        if (overlap(pk, act, residual, act) || overlap(pk, act, weight, wb) || overlap(pk, act, out, outb) ||
            (dyn && overlap(pk, act, scale, sb)) || (fp4 && overlap(pk, act, out_sf, sfb)))
            return MBD_ERR_INVALID_ARG;
    }

    p->x = x;
    p->n_partials = partials ? n_partials : 0;
    for (int k = 0; k < p->n_partials; ++k) p->partials[k] = partials[k];
    p->residual = residual;
    p->weight = weight;
    p->out = out;
    p->out_sf = out_sf;
    p->scale = scale;
    p->rows = n_tokens;
    p->nvec = static_cast<int>(hidden / 8);
    p->hidden = static_cast<int>(hidden);
    p->eps = eps;
    return MBD_OK;
}

// ------------------------------------------------------------------------------------------ tuning table

// The shape-bucket dispatch table (mbd_tuning_set): an immutable vector swapped in whole, so a call reads a
// consistent table without locking while another thread replaces it.
std::shared_ptr<const std::vector<mbd_tuning_entry>> g_tuning;

std::shared_ptr<const std::vector<mbd_tuning_entry>> tuning_table() { return std::atomic_load(&g_tuning); }

bool valid_kind_mode(int kind, int mode) {
    if (kind < MBD_OP_ADD_RMSNORM || kind > MBD_OP_SWIGLU_QUANT_NVFP4) return false;
    const bool fp8 = kind == MBD_OP_ADD_RMSNORM_QUANT_FP8 || kind == MBD_OP_SWIGLU_QUANT_FP8;
    return !fp8 || mode == MBD_SCALE_STATIC_PER_TENSOR || mode == MBD_SCALE_DYNAMIC_PER_TOKEN;
}

// The launch shape of an entry, made concrete for one call, or false if it does not fit the call (then the
// built-in rules decide). The same legality as the rules' shapes: at most 8 CTAs (one cluster) when the row
// is reduced, slices covering the row, even slices for NVFP4.
bool entry_plan(const mbd_tuning_entry& e, int64_t rows, int nvec, bool reduces, bool pairs, int sms,
                mbd::RowPlan* plan) {
    const int v = e.vectors_per_thread, th = e.threads;
    if (e.ctas_per_row < 1 || (reduces && e.ctas_per_row > 8)) return false;
    if (!(v == 1 || v == 2 || v == 4 || v == 8) || th < 32 || th > 512 || th % 32 != 0) return false;
    int slice = cdiv(nvec, e.ctas_per_row);
    if (pairs && (slice & 1)) ++slice;
    const int c = cdiv(nvec, slice);
    if (int64_t{th} * v < slice || rows > mbd::kMaxGridYZ * mbd::kMaxGridYZ) return false;
    *plan = mbd::RowPlan{};
    plan->ctas_per_row = c;
    plan->slice = slice;
    plan->threads = th;
    plan->vpt = v;
    plan->prefetch = rows < sms ? 1 : 0;
    return true;
}

// The wave-ahead L2 warming of the rules, for a plan that came from the table.
void set_ahead(bool dyn_swiglu, int64_t rows, int sms, mbd::RowPlan* plan) {
    if (dyn_swiglu && rows >= 4 * int64_t{sms} && plan->vpt <= 2)
        plan->ahead = static_cast<int>(int64_t{sms} * (2048 / plan->threads) / plan->ctas_per_row / 2);
}

// Large batches of wide dynamic-FP8 SwiGLU rows: the slices come into shared memory by bulk copies and
// registers hold only the products (swiglu_dyn_bulk_kernel), 5 CTAs of 256 threads per SM. Clusters of 7
// (8 past 7 x 1280 vectors), 4 vectors per thread, L2 warmed half the resident rows ahead. Measured at
// 4 or more rows per SM (CUDA events around back-to-back launches, inputs > L2, bit-identical outputs):
// I 53248: 82.6 vs 87.5 us at T 2048 (clusters of 8: 88.2, of 6: 85.7), 158.5 vs 168.8 at T 4096; at
// I 28672 the register form stays ahead (85.1 vs 87.0 us at T 4096, best bulk shape), likewise at I 13824,
// so rows of up to 4608 vectors keep it. It supersedes table entries for the shapes it takes.
constexpr int kBulkMinVec = 4609, kBulkMaxSlice = 1280;   // kBulkMaxSlice: 320 threads x 4 vectors
void bulk_rule(int64_t rows, int nvec, int sms, mbd::RowPlan* plan) {
    if (rows < 4 * int64_t{sms} || nvec < kBulkMinVec || nvec > 8 * kBulkMaxSlice) return;
    int c = cdiv(nvec, kBulkMaxSlice);
    if (c < 7) c = 7;
    const int slice = cdiv(nvec, c);
    *plan = mbd::RowPlan{};
    plan->ctas_per_row = cdiv(nvec, slice);
    plan->slice = slice;
    plan->vpt = 4;
    plan->threads = cdiv(cdiv(slice, 4), 32) * 32;
    plan->bulk = 1;
    plan->ahead = static_cast<int>(int64_t{sms} * 5 / plan->ctas_per_row / 2);
}

// The first table entry whose buckets hold the call and whose shape fits it.
bool tuned_plan(int kind, int mode, int64_t rows, int64_t width, int nvec, bool reduces, bool pairs, int sms,
                mbd::RowPlan* plan) {
    const auto table = tuning_table();
    if (!table) return false;
    const bool fp8 = kind == MBD_OP_ADD_RMSNORM_QUANT_FP8 || kind == MBD_OP_SWIGLU_QUANT_FP8;
    for (const mbd_tuning_entry& e : *table) {
        if (e.kind != kind || (fp8 && e.mode != mode)) continue;
        if (rows < e.tokens_min || rows > e.tokens_max || width < e.width_min || width > e.width_max) continue;
        if (entry_plan(e, rows, nvec, reduces, pairs, sms, plan)) return true;
    }
    return false;
}

int norm_kind(mbd::Epilogue ep) {
    return ep == mbd::kBf16 ? MBD_OP_ADD_RMSNORM
                            : (ep == mbd::kNvfp4 ? MBD_OP_ADD_RMSNORM_QUANT_NVFP4 : MBD_OP_ADD_RMSNORM_QUANT_FP8);
}
int swiglu_kind(mbd::Epilogue ep) {
    return ep == mbd::kBf16 ? MBD_OP_SWIGLU : (ep == mbd::kNvfp4 ? MBD_OP_SWIGLU_QUANT_NVFP4 : MBD_OP_SWIGLU_QUANT_FP8);
}
int scale_mode(mbd::Epilogue ep) { return ep == mbd::kFp8Dynamic ? MBD_SCALE_DYNAMIC_PER_TOKEN : MBD_SCALE_STATIC_PER_TENSOR; }

// The launch shape of a prepared norm call (the table, else the rules); false if none fits.
bool norm_plan(const mbd::NormParams& p, mbd::Epilogue ep, int sms, mbd::RowPlan* plan) {
    const bool partials = p.n_partials > 0;
    const bool tuned = !partials && tuned_plan(norm_kind(ep), scale_mode(ep), p.rows, p.hidden, p.nvec, true,
                                                ep == mbd::kNvfp4, sms, plan);
    return tuned ||
           plan_rows(p.rows, p.nvec, partials ? Shape::kNormPartials : Shape::kNorm, sms, ep == mbd::kNvfp4, plan);
}

mbd_status norm_common(void* out, uint8_t* out_sf, mbd::Epilogue ep, void* residual, const void* x,
                       const void* weight, int64_t n_tokens, int64_t hidden, float eps, float* scale,
                       cudaStream_t stream, const void* const* partials = nullptr, int n_partials = 0) {
    mbd::NormParams p;
    const mbd_status st =
        norm_prepare(out, out_sf, ep, residual, x, weight, n_tokens, hidden, eps, scale, partials, n_partials, &p);
    if (st != MBD_OK || p.rows == 0) return st;
    mbd::RowPlan plan;
    if (!norm_plan(p, ep, sm_count_of_current_device(), &plan)) return MBD_ERR_UNSUPPORTED;
    return finish_launch(mbd::launch_add_rmsnorm(p, ep, plan, stream));
}

mbd_status swiglu_prepare(void* out, uint8_t* out_sf, mbd::Epilogue ep, const void* gate_up, int64_t n_tokens,
                          int64_t inter, float* scale, mbd::SwigluParams* p) {
    *p = mbd::SwigluParams{};
    mbd_status st = check_width(n_tokens, inter);
    if (st != MBD_OK) return st;
    const bool quant = ep != mbd::kBf16, dyn = ep == mbd::kFp8Dynamic, fp4 = ep == mbd::kNvfp4;
    if (fp4 && inter % 16 != 0) return MBD_ERR_MISALIGNED;
    if (dyn && inter > MBD_MAX_REDUCED_WIDTH) return MBD_ERR_UNSUPPORTED;
    if (n_tokens == 0) return MBD_OK;
    if (!out || !gate_up || (quant && !scale) || (fp4 && !out_sf)) return MBD_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(gate_up, 16) || (quant && !aligned(scale, 4))) return MBD_ERR_MISALIGNED;
    const size_t inb = static_cast<size_t>(n_tokens) * static_cast<size_t>(inter) * 4;
    const size_t outb = out_bytes(ep, n_tokens, inter);
    const size_t sfb = fp4 ? static_cast<size_t>(n_tokens) * static_cast<size_t>(inter / 16) : 0;
    const size_t sb = quant ? (dyn ? static_cast<size_t>(n_tokens) * 4 : 4) : 0;
    if (overlap(out, outb, gate_up, inb)) return MBD_ERR_INVALID_ARG;
    if (quant && overlap(scale, sb, out, outb)) return MBD_ERR_INVALID_ARG;
    if (dyn && overlap(scale, sb, gate_up, inb)) return MBD_ERR_INVALID_ARG;
    if (fp4 && (overlap(out_sf, sfb, out, outb) || overlap(out_sf, sfb, gate_up, inb) ||
                overlap(out_sf, sfb, scale, sb)))
        return MBD_ERR_INVALID_ARG;

    *p = mbd::SwigluParams{gate_up, out, scale, n_tokens, static_cast<int>(inter / 8), out_sf};
    return MBD_OK;
}

// The launch shape of a prepared SwiGLU call (the table, else the rules; the bulk-copy rule last); false if
// none fits.
bool swiglu_plan(const mbd::SwigluParams& p, mbd::Epilogue ep, int sms, mbd::RowPlan* plan) {
    const int64_t inter = int64_t{p.nvec} * 8;
    const bool tuned = tuned_plan(swiglu_kind(ep), scale_mode(ep), p.rows, inter, p.nvec, ep == mbd::kFp8Dynamic,
                                  ep == mbd::kNvfp4, sms, plan);
    if (tuned) set_ahead(ep == mbd::kFp8Dynamic, p.rows, sms, plan);
    if (!tuned && !plan_rows(p.rows, p.nvec, ep == mbd::kFp8Dynamic ? Shape::kRowMax : Shape::kStream, sms,
                             ep == mbd::kNvfp4, plan))
        return false;
    if (ep == mbd::kFp8Dynamic) bulk_rule(p.rows, p.nvec, sms, plan);
    return true;
}

mbd_status swiglu_common(void* out, uint8_t* out_sf, mbd::Epilogue ep, const void* gate_up, int64_t n_tokens,
                         int64_t inter, float* scale, cudaStream_t stream) {
    mbd::SwigluParams p;
    const mbd_status st = swiglu_prepare(out, out_sf, ep, gate_up, n_tokens, inter, scale, &p);
    if (st != MBD_OK || p.rows == 0) return st;
    mbd::RowPlan plan;
    if (!swiglu_plan(p, ep, sm_count_of_current_device(), &plan)) return MBD_ERR_UNSUPPORTED;
    return finish_launch(mbd::launch_swiglu(p, ep, plan, stream));
}

// ------------------------------------------------------------------------------------------ programs

static_assert(sizeof(mbd::ProgramParams) <= 32764, "program parameters exceed the kernel parameter limit");
static_assert(mbd::kMaxProgramOps == MBD_MAX_PROGRAM_OPS, "program op limit");
static_assert(mbd::kStaticScheduleBytes == MBD_STATIC_SCHEDULE_BYTES, "static schedule size");
static_assert(sizeof(mbd_op) == 80 && offsetof(mbd_op, out) == 32 && offsetof(mbd_op, scale) == 72, "mbd_op layout");

// A byte range an op touches: row-wise ranges (row_bytes > 0) hold `rows` rows of row_bytes each.
struct Region {
    const void* ptr;
    size_t bytes;
    bool write;
    size_t row_bytes;
    int64_t rows;
};

struct OpInfo {
    Region reg[6];
    int nreg;
    bool holds_row;   // reduces over its row: the whole row stays in one CTA
};

void add_region(OpInfo& o, const void* ptr, size_t bytes, bool write, size_t row_bytes, int64_t rows) {
    if (ptr && bytes) o.reg[o.nreg++] = Region{ptr, bytes, write, row_bytes, rows};
}

// Union-find over op indices; unions keep the smaller index as the root, so a chain's root is its first op.
int find_root(int* parent, int i) {
    while (parent[i] != i) i = parent[i] = parent[parent[i]];
    return i;
}

// Resident program CTAs per SM, queried once per device, vectors per thread and variant.
std::atomic<int> g_prog_ctas[kMaxDevices][4][mbd::kProgramVariants];

int program_ctas_per_sm_cached(int vpt, int variant) {
    int dev = 0;
    const int vi = vpt == 1 ? 0 : (vpt == 2 ? 1 : (vpt == 4 ? 2 : 3));
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return mbd::program_ctas_per_sm(vpt, variant);
    }
    int n = g_prog_ctas[dev][vi][variant].load(std::memory_order_relaxed);
    if (n > 0) return n;
    n = mbd::program_ctas_per_sm(vpt, variant);
    if (n > 0) g_prog_ctas[dev][vi][variant].store(n, std::memory_order_relaxed);
    return n;
}

// A built program: the kernel's parameters and its launch shape, for the device it was built on.
struct PlanImpl {
    uint32_t magic;
    int device;
    int vpt, variant, grid, pad;
    mbd::ProgramParams P;
};
constexpr uint32_t kPlanMagic = 0x4d424450u;
static_assert(sizeof(PlanImpl) <= sizeof(mbd_program_plan), "program plan size");
static_assert(alignof(PlanImpl) <= alignof(mbd_program_plan), "program plan alignment");

mbd_status build_program(const mbd_op* ops, int n_ops, PlanImpl* plan) {
    if (!plan) return MBD_ERR_INVALID_ARG;
    plan->magic = 0;
    if (n_ops < 0 || n_ops > MBD_MAX_PROGRAM_OPS || (n_ops > 0 && !ops)) return MBD_ERR_INVALID_ARG;
    int device = -1;   // queried once there is something to launch (every check before it is host-only)
    mbd::ProgramParams& P = plan->P;
    P = mbd::ProgramParams{};
    P.n_ops = n_ops;
    OpInfo info[MBD_MAX_PROGRAM_OPS];
    bool active[MBD_MAX_PROGRAM_OPS] = {};
    int norm_mask = 0, swiglu_mask = 0, max_held_nvec = 0, max_dyn_nvec = 0;
    for (int i = 0; i < n_ops; ++i) {
        const mbd_op& o = ops[i];
        if (o.reserved != 0 || o.kind < MBD_OP_ADD_RMSNORM || o.kind > MBD_OP_SWIGLU_QUANT_NVFP4) return MBD_ERR_INVALID_ARG;
        const bool is_norm = o.kind <= MBD_OP_ADD_RMSNORM_QUANT_NVFP4;
        const int sub = is_norm ? o.kind : o.kind - MBD_OP_SWIGLU;   // 0 bf16, 1 FP8, 2 NVFP4
        mbd::Epilogue ep = sub == 0 ? mbd::kBf16 : mbd::kNvfp4;
        if (sub == 1 && !fp8_epilogue(o.mode, &ep)) return MBD_ERR_INVALID_ARG;
        mbd::ProgOp& po = P.ops[i];
        OpInfo& in = info[i];
        in.nreg = 0;
        const size_t W = static_cast<size_t>(o.width);
        if (is_norm) {
            mbd::NormParams np;
            const mbd_status st = norm_prepare(o.out, o.out_sf, ep, o.residual, o.in, o.weight, o.n_tokens, o.width,
                                               o.eps, o.scale, nullptr, 0, &np);
            if (st != MBD_OK) return st;
            if (np.rows == 0) continue;
            po = mbd::ProgOp{np.x, np.residual, np.weight, np.out, np.out_sf, np.scale, np.rows, mbd::kOpNorm,
                             ep, np.nvec, np.hidden, np.eps, 0};
            add_region(in, o.in, np.rows * W * 2, false, W * 2, np.rows);
            add_region(in, o.residual, np.rows * W * 2, true, W * 2, np.rows);
            add_region(in, o.weight, W * 2, false, 0, 0);
            in.holds_row = true;
            norm_mask |= 1 << ep;
        } else {
            mbd::SwigluParams sp;
            const mbd_status st = swiglu_prepare(o.out, o.out_sf, ep, o.in, o.n_tokens, o.width, o.scale, &sp);
            if (st != MBD_OK) return st;
            if (sp.rows == 0) continue;
            po = mbd::ProgOp{sp.gate_up, nullptr, nullptr, sp.out, sp.out_sf, sp.scale, sp.rows, mbd::kOpSwiglu, ep,
                             sp.nvec, static_cast<int>(o.width), 0.0f, 0};
            add_region(in, o.in, sp.rows * W * 4, false, W * 4, sp.rows);
            in.holds_row = false;   // streams run in chunks; a wide dynamic row takes two passes
            swiglu_mask |= 1 << ep;
            if (ep == mbd::kFp8Dynamic && sp.nvec > max_dyn_nvec) max_dyn_nvec = sp.nvec;
        }
        const int64_t T = po.rows;
        const size_t out_row = ep == mbd::kBf16 ? 2 * W : (ep == mbd::kNvfp4 ? W / 2 : W);
        add_region(in, o.out, T * out_row, true, out_row, T);
        if (ep == mbd::kNvfp4) add_region(in, o.out_sf, T * (W / 16), true, W / 16, T);
        if (ep == mbd::kFp8Dynamic) add_region(in, o.scale, T * 4, true, 4, T);
        else if (ep != mbd::kBf16) add_region(in, o.scale, 4, false, 0, 0);
        if (in.holds_row && po.nvec > max_held_nvec) max_held_nvec = po.nvec;
        active[i] = true;
    }
    // ops linked by a shared, written buffer form chains (union-find over the overlapping pairs of regions,
    // found by sorting all regions by start address and sweeping)
    int parent[MBD_MAX_PROGRAM_OPS];
    for (int i = 0; i < n_ops; ++i) parent[i] = i;
    struct RegRef {
        uintptr_t lo, hi;
        int op, reg;
    };
    RegRef refs[MBD_MAX_PROGRAM_OPS * 6];
    int nref = 0;
    for (int i = 0; i < n_ops; ++i)
        for (int q = 0; active[i] && q < info[i].nreg; ++q) {
            const uintptr_t lo = reinterpret_cast<uintptr_t>(info[i].reg[q].ptr);
            refs[nref++] = RegRef{lo, lo + info[i].reg[q].bytes, i, q};
        }
    std::sort(refs, refs + nref, [](const RegRef& a, const RegRef& b) { return a.lo < b.lo; });
    int open_refs[MBD_MAX_PROGRAM_OPS * 6];
    int nopen = 0;
    for (int r = 0; r < nref; ++r) {
        int keep = 0;   // drop the regions that end before this one starts
        for (int k = 0; k < nopen; ++k)
            if (refs[open_refs[k]].hi > refs[r].lo) open_refs[keep++] = open_refs[k];
        nopen = keep;
        const Region& y = info[refs[r].op].reg[refs[r].reg];
        for (int k = 0; k < nopen; ++k) {
            const RegRef& a = refs[open_refs[k]];
            if (a.op == refs[r].op) continue;   // within one op: checked by its entry point's rules
            const Region& x = info[a.op].reg[a.reg];
            if (!(x.write || y.write)) continue;
            if (!(x.row_bytes > 0 && x.ptr == y.ptr && x.row_bytes == y.row_bytes && x.rows == y.rows))
                return MBD_ERR_UNSUPPORTED;
            const int ra = find_root(parent, a.op), rb = find_root(parent, refs[r].op);
            parent[ra > rb ? ra : rb] = ra < rb ? ra : rb;   // the root stays the chain's first op
        }
        open_refs[nopen++] = r;
    }
    int size[MBD_MAX_PROGRAM_OPS] = {};
    for (int i = 0; i < n_ops; ++i)
        if (active[i]) ++size[find_root(parent, i)];
    if (max_held_nvec > MBD_MAX_PROGRAM_WIDTH / 8) return MBD_ERR_UNSUPPORTED;
    int vpt = max_held_nvec <= mbd::kProgramThreads ? 1 : (max_held_nvec <= 2 * mbd::kProgramThreads ? 2 : 4);
    const int variant = mbd::program_variant(norm_mask, swiglu_mask);
    if (variant < 0) return MBD_ERR_UNSUPPORTED;
    // A dynamic-FP8 SwiGLU row wider than the CTA holds at this vpt runs in two passes (each a memory round
    // trip, the products computed twice); up to 8 vectors per thread it runs in one at vpt 8. Except where
    // the chains' norms run with the residual row in registers (vpt 1, one norm epilogue): a decode step's
    // chained norms are its critical path, and its SwiGLU rows run beside them.
    bool has_chain = false;
    for (int i = 0; i < n_ops; ++i) has_chain |= active[i] && find_root(parent, i) == i && size[i] > 1;
    if (max_dyn_nvec > mbd::kProgramThreads * vpt && max_dyn_nvec <= 8 * mbd::kProgramThreads &&
        mbd::program_variant_has_vpt8(variant) && !(has_chain && mbd::program_norms_in_registers(vpt, variant)))
        vpt = 8;
    P.chunk_vecs = mbd::kProgramThreads * (vpt < 4 ? vpt : 4);

    // chains in the order of their first op, each op after the ops before it in the list
    int order_len = 0;
    int64_t warm_row_bytes = 0;
    for (int r = 0; r < n_ops; ++r) {
        if (!active[r] || find_root(parent, r) != r) continue;
        if (size[r] > 1) {
            P.group_begin[P.n_groups] = order_len;
            P.group_items[P.n_groups] = P.n_chain_items;
            for (int i = r; i < n_ops; ++i) {
                if (!active[i] || find_root(parent, i) != r) continue;
                // warm this op's row inputs unless an earlier op of the chain writes them
                mbd::ProgOp& po = P.ops[i];
                bool in_written = false, res_written = false;
                for (int k = P.group_begin[P.n_groups]; k < order_len; ++k)
                    for (int q = 0; q < info[P.chain_order[k]].nreg; ++q) {
                        const Region& w = info[P.chain_order[k]].reg[q];
                        if (!w.write) continue;
                        in_written |= overlap(w.ptr, w.bytes, po.in, static_cast<size_t>(po.rows) * po.nvec *
                                                                         (po.cls == mbd::kOpNorm ? 16 : 32));
                        if (po.residual)
                            res_written |= overlap(w.ptr, w.bytes, po.residual, static_cast<size_t>(po.rows) * po.nvec * 16);
                    }
                po.prefetch = (in_written ? 0 : 1) | ((po.residual && !res_written) ? 2 : 0);
                if (order_len > P.group_begin[P.n_groups]) {   // continues a run of norms on one residual row
                    const mbd::ProgOp& prev = P.ops[P.chain_order[order_len - 1]];
                    if (po.cls == mbd::kOpNorm && prev.cls == mbd::kOpNorm && po.residual == prev.residual &&
                        po.nvec == prev.nvec && po.rows == prev.rows && !in_written)
                        po.prefetch |= mbd::kContinuesRun;
                }
                warm_row_bytes += (in_written ? 0 : int64_t{po.nvec} * (po.cls == mbd::kOpNorm ? 16 : 32)) +
                                  ((po.residual && !res_written) ? int64_t{po.nvec} * 16 : 0);
                P.chain_order[order_len++] = i;
            }
            P.n_chain_items += P.ops[r].rows;
            ++P.n_groups;
        } else {
            P.free_op[P.n_free] = r;
            P.free_chunks[P.n_free] = (info[r].holds_row || P.ops[r].ep == mbd::kFp8Dynamic)
                                          ? 1 : cdiv(P.ops[r].nvec, P.chunk_vecs);
            P.free_items[P.n_free] = P.n_free_items;
            P.n_free_items += P.ops[r].rows * P.free_chunks[P.n_free];
            ++P.n_free;
        }
    }
    P.group_begin[P.n_groups] = order_len;
    P.group_items[P.n_groups] = P.n_chain_items;
    P.free_items[P.n_free] = P.n_free_items;
    const int64_t items = P.n_chain_items + P.n_free_items;
    int grid = 0;
    if (items > 0) {
        if (cudaGetDevice(&device) != cudaSuccess) {
            g_last_cuda_error = static_cast<int>(cudaGetLastError());
            return MBD_ERR_CUDA;
        }
        const int per_sm = program_ctas_per_sm_cached(vpt, variant);
        if (per_sm <= 0) {
            g_last_cuda_error = static_cast<int>(cudaErrorInvalidConfiguration);
            return MBD_ERR_CUDA;
        }
        const int64_t slots = int64_t{sm_count_of_current_device()} * per_sm;
        grid = static_cast<int>(items < slots ? items : slots);
        // warm the chains' row inputs only while the rows in flight fit well inside L2 (a quarter of 126 MiB)
        P.prefetch_chains = warm_row_bytes * (P.n_chain_items < grid ? P.n_chain_items : grid) <= (int64_t{32} << 20);
    }
    plan->device = device;
    plan->vpt = vpt;
    plan->variant = variant;
    plan->grid = grid;
    plan->pad = 0;
    plan->magic = kPlanMagic;
    return MBD_OK;
}

mbd_status launch_plan(const PlanImpl* plan, cudaStream_t stream) {
    if (!plan || plan->magic != kPlanMagic) return MBD_ERR_INVALID_ARG;
    if (plan->grid == 0) return MBD_OK;   // nothing to do
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) {
        g_last_cuda_error = static_cast<int>(cudaGetLastError());
        return MBD_ERR_CUDA;
    }
    if (device != plan->device) return MBD_ERR_INVALID_ARG;
    return finish_launch(mbd::launch_program(plan->P, nullptr, plan->vpt, plan->variant, plan->grid, stream));
}

constexpr size_t kScheduleBytes = (sizeof(mbd::ProgramParams) + 255) & ~size_t{255};

mbd_status upload_plan(const PlanImpl* plan, void* schedule, size_t bytes, cudaStream_t stream) {
    if (!plan || plan->magic != kPlanMagic || !schedule) return MBD_ERR_INVALID_ARG;
    if (!aligned(schedule, 256)) return MBD_ERR_MISALIGNED;
    if (bytes < kScheduleBytes) return MBD_ERR_INVALID_ARG;
    const cudaError_t e = cudaMemcpyAsync(schedule, &plan->P, sizeof(mbd::ProgramParams), cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) {
        g_last_cuda_error = static_cast<int>(e);
        (void)cudaGetLastError();
        return MBD_ERR_CUDA;
    }
    return MBD_OK;
}

mbd_status launch_uploaded(const PlanImpl* plan, const void* schedule, cudaStream_t stream) {
    if (!plan || plan->magic != kPlanMagic || !schedule) return MBD_ERR_INVALID_ARG;
    if (!aligned(schedule, 256)) return MBD_ERR_MISALIGNED;
    if (plan->grid == 0) return MBD_OK;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) {
        g_last_cuda_error = static_cast<int>(cudaGetLastError());
        return MBD_ERR_CUDA;
    }
    if (device != plan->device) return MBD_ERR_INVALID_ARG;
    return finish_launch(mbd::launch_program(plan->P, static_cast<const mbd::ProgramParams*>(schedule), plan->vpt,
                                             plan->variant, plan->grid, stream));
}

static_assert(kScheduleBytes <= mbd::kStaticScheduleBytes, "every schedule record fits the static buffer");

// mbd_program_plan_launch_static: the uploaded-schedule launch, with the schedule copied into the static
// buffer instead of caller memory. Nothing is allocated: the buffer is part of the module image.
mbd_status launch_static(const PlanImpl* plan, cudaStream_t stream) {
    if (!plan || plan->magic != kPlanMagic) return MBD_ERR_INVALID_ARG;
    if (plan->grid == 0) return MBD_OK;
    int device = 0;
    const cudaError_t de = cudaGetDevice(&device);
    if (de != cudaSuccess || device < 0 || device >= mbd::kMaxCachedDevices) {
        g_last_cuda_error = static_cast<int>(de != cudaSuccess ? de : cudaErrorInvalidDevice);
        (void)cudaGetLastError();
        return MBD_ERR_CUDA;
    }
    if (device != plan->device) return MBD_ERR_INVALID_ARG;
    void* addr = nullptr;
    const cudaError_t e = mbd::static_schedule_address(device, &addr);
    if (e != cudaSuccess) {
        g_last_cuda_error = static_cast<int>(e);
        (void)cudaGetLastError();
        return MBD_ERR_CUDA;
    }
    const mbd_status st = upload_plan(plan, addr, mbd::kStaticScheduleBytes, stream);
    if (st != MBD_OK) return st;
    return launch_uploaded(plan, addr, stream);
}

// ------------------------------------------------------------------------------------------ batches

// The byte ranges one op of a program touches (for the independence check of a batch it opens).
OpInfo prog_op_regions(const mbd::ProgOp& op) {
    OpInfo in;
    in.nreg = 0;
    in.holds_row = false;
    if (op.rows <= 0) return in;
    const size_t T = static_cast<size_t>(op.rows), V = static_cast<size_t>(op.nvec);
    if (op.cls == mbd::kOpNorm) {
        add_region(in, op.in, T * V * 16, false, 0, 0);
        add_region(in, op.residual, T * V * 16, true, 0, 0);
        add_region(in, op.weight, V * 16, false, 0, 0);
    } else {
        add_region(in, op.in, T * V * 32, false, 0, 0);
    }
    const size_t out_row = op.ep == mbd::kBf16 ? V * 16 : (op.ep == mbd::kNvfp4 ? V * 4 : V * 8);
    add_region(in, op.out, T * out_row, true, 0, 0);
    if (op.ep == mbd::kNvfp4) add_region(in, op.out_sf, T * (V / 2), true, 0, 0);
    if (op.ep == mbd::kFp8Dynamic) add_region(in, op.scale, T * 4, true, 0, 0);
    else if (op.ep != mbd::kBf16) add_region(in, op.scale, 4, false, 0, 0);
    return in;
}

bool conflict(const OpInfo& x, const OpInfo& y) {   // one writes what the other reads or writes
    for (int u = 0; u < x.nreg; ++u)
        for (int v = 0; v < y.nreg; ++v)
            if ((x.reg[u].write || y.reg[v].write) && overlap(x.reg[u].ptr, x.reg[u].bytes, y.reg[v].ptr, y.reg[v].bytes))
                return true;
    return false;
}

// mbd_run_independent[_with_program]: ops that share no written memory, each launched as its single call, and
// optionally a program (uploaded schedule) in front of them. The first launch takes PdlOrder kPdlHead (the
// program: its early trigger), the rest kPdlOverlap. Every op is checked, and then planned, before the first
// launch.
mbd_status run_independent(const PlanImpl* plan, const void* schedule, const mbd_op* ops, int n_ops,
                           cudaStream_t stream) {
    if (n_ops < 0 || n_ops > MBD_MAX_INDEPENDENT_OPS || (n_ops > 0 && !ops)) return MBD_ERR_INVALID_ARG;
    if (plan) {
        if (plan->magic != kPlanMagic || !schedule) return MBD_ERR_INVALID_ARG;
        if (!aligned(schedule, 256)) return MBD_ERR_MISALIGNED;
    }
    struct Prepared {
        bool norm;
        mbd::Epilogue ep;
        mbd::NormParams np;
        mbd::SwigluParams sp;
        OpInfo info;
    };
    Prepared prep[MBD_MAX_INDEPENDENT_OPS];
    int active[MBD_MAX_INDEPENDENT_OPS];
    int n_active = 0;
    for (int i = 0; i < n_ops; ++i) {
        const mbd_op& o = ops[i];
        if (o.reserved != 0 || o.kind < MBD_OP_ADD_RMSNORM || o.kind > MBD_OP_SWIGLU_QUANT_NVFP4) return MBD_ERR_INVALID_ARG;
        Prepared& q = prep[i];
        q.norm = o.kind <= MBD_OP_ADD_RMSNORM_QUANT_NVFP4;
        const int sub = q.norm ? o.kind : o.kind - MBD_OP_SWIGLU;   // 0 bf16, 1 FP8, 2 NVFP4
        q.ep = sub == 0 ? mbd::kBf16 : mbd::kNvfp4;
        if (sub == 1 && !fp8_epilogue(o.mode, &q.ep)) return MBD_ERR_INVALID_ARG;
        q.info.nreg = 0;
        const size_t W = static_cast<size_t>(o.width);
        int64_t T = 0;
        if (q.norm) {
            const mbd_status st = norm_prepare(o.out, o.out_sf, q.ep, o.residual, o.in, o.weight, o.n_tokens, o.width,
                                               o.eps, o.scale, nullptr, 0, &q.np);
            if (st != MBD_OK) return st;
            T = q.np.rows;
            add_region(q.info, o.in, T * W * 2, false, 0, 0);
            add_region(q.info, o.residual, T * W * 2, true, 0, 0);
            add_region(q.info, o.weight, W * 2, false, 0, 0);
        } else {
            const mbd_status st = swiglu_prepare(o.out, o.out_sf, q.ep, o.in, o.n_tokens, o.width, o.scale, &q.sp);
            if (st != MBD_OK) return st;
            T = q.sp.rows;
            add_region(q.info, o.in, T * W * 4, false, 0, 0);
        }
        if (T == 0) continue;   // nothing to do, nothing touched
        add_region(q.info, o.out, out_bytes(q.ep, T, o.width), true, 0, 0);
        if (q.ep == mbd::kNvfp4) add_region(q.info, o.out_sf, T * (W / 16), true, 0, 0);
        if (q.ep == mbd::kFp8Dynamic) add_region(q.info, o.scale, T * 4, true, 0, 0);
        else if (q.ep != mbd::kBf16) add_region(q.info, o.scale, 4, false, 0, 0);
        active[n_active++] = i;
    }
    // independence: what one op writes, no other op may read or write (the program's ops among themselves are
    // the program's business)
    for (int a = 0; a < n_active; ++a)
        for (int b = a + 1; b < n_active; ++b)
            if (conflict(prep[active[a]].info, prep[active[b]].info)) return MBD_ERR_INVALID_ARG;
    const bool with_program = plan && plan->grid > 0;
    if (with_program) {
        for (int k = 0; k < plan->P.n_ops; ++k) {
            const OpInfo pi = prog_op_regions(plan->P.ops[k]);
            if (pi.nreg == 0) continue;
            for (int a = 0; a < n_active; ++a)
                if (conflict(pi, prep[active[a]].info)) return MBD_ERR_INVALID_ARG;
        }
        int device = 0;
        const cudaError_t de = cudaGetDevice(&device);
        if (de != cudaSuccess) {
            g_last_cuda_error = static_cast<int>(de);
            (void)cudaGetLastError();
            return MBD_ERR_CUDA;
        }
        if (device != plan->device) return MBD_ERR_INVALID_ARG;
    }
    if (n_active == 0 && !with_program) return MBD_OK;
    const int sms = sm_count_of_current_device();
    mbd::RowPlan plans[MBD_MAX_INDEPENDENT_OPS];
    for (int a = 0; a < n_active; ++a) {
        const Prepared& q = prep[active[a]];
        if (!(q.norm ? norm_plan(q.np, q.ep, sms, &plans[a]) : swiglu_plan(q.sp, q.ep, sms, &plans[a])))
            return MBD_ERR_UNSUPPORTED;
        plans[a].order = (a == 0 && !with_program) ? mbd::kPdlHead : mbd::kPdlOverlap;
    }
    // The program first (measured on the 405B step's twelve small calls beside five large ones: 169.4 us per
    // step with the program first, 170.1 with it last, where its CTAs wait for SMs the ops' last wave frees)
    if (with_program) {
        const mbd_status st = finish_launch(mbd::launch_program(plan->P, static_cast<const mbd::ProgramParams*>(schedule),
                                                                plan->vpt, plan->variant, plan->grid, stream,
                                                                mbd::kPdlHead));
        if (st != MBD_OK) return st;
    }
    for (int a = 0; a < n_active; ++a) {
        const Prepared& q = prep[active[a]];
        const mbd_status st = finish_launch(q.norm ? mbd::launch_add_rmsnorm(q.np, q.ep, plans[a], stream)
                                                   : mbd::launch_swiglu(q.sp, q.ep, plans[a], stream));
        if (st != MBD_OK) return st;
    }
    return MBD_OK;
}

}  // namespace

extern "C" {

int mbd_abi_version(void) { return MBD_ABI_VERSION; }

const char* mbd_status_string(int status) {
    switch (status) {
        case MBD_OK: return "MBD_OK";
        case MBD_ERR_INVALID_ARG: return "MBD_ERR_INVALID_ARG: invalid argument";
        case MBD_ERR_MISALIGNED: return "MBD_ERR_MISALIGNED: pointer or width not aligned to 16 bytes";
        case MBD_ERR_UNSUPPORTED: return "MBD_ERR_UNSUPPORTED: shape beyond the library's limits";
        case MBD_ERR_CUDA: return "MBD_ERR_CUDA: kernel launch failed (see mbd_last_cuda_error)";
        default: return "unknown mbd_status";
    }
}

int mbd_last_cuda_error(void) { return g_last_cuda_error; }

uint64_t mbd_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

mbd_status mbd_device_error_flags(uint32_t* flags, int clear) {
    if (!flags) return MBD_ERR_INVALID_ARG;
    unsigned int a = 0, b = 0, c = 0;
    cudaError_t e = mbd::device_error_flags_norm(&a, clear != 0);
    if (e == cudaSuccess) e = mbd::device_error_flags_swiglu(&b, clear != 0);
    if (e == cudaSuccess) e = mbd::device_error_flags_selftest(&c, clear != 0);
    unsigned int d = 0;
    if (e == cudaSuccess) e = mbd::device_error_flags_program(&d, clear != 0);
    if (e != cudaSuccess) {
        g_last_cuda_error = static_cast<int>(e);
        (void)cudaGetLastError();
        return MBD_ERR_CUDA;
    }
    *flags = a | b | c | d;
    return MBD_OK;
}

mbd_status mbd_selftest_bounded_wait(uint64_t limit_cycles, mbd_stream_t stream) {
    if (limit_cycles == 0 || limit_cycles > (uint64_t{1} << 31)) return MBD_ERR_INVALID_ARG;
    const cudaError_t e =
        mbd::launch_bounded_wait_probe(static_cast<long long>(limit_cycles), reinterpret_cast<cudaStream_t>(stream));
    return finish_launch(e);
}

mbd_status mbd_fused_add_rmsnorm(void* out, void* residual, const void* x, const void* weight,
                                 int64_t n_tokens, int64_t hidden, float eps, mbd_stream_t stream) {
    return norm_common(out, nullptr, mbd::kBf16, residual, x, weight, n_tokens, hidden, eps, nullptr,
                       reinterpret_cast<cudaStream_t>(stream));
}

mbd_status mbd_fused_add_rmsnorm_quant_fp8(uint8_t* out_q, void* residual, const void* x,
                                           const void* weight, int64_t n_tokens, int64_t hidden, float eps,
                                           mbd_scale_mode mode, float* scale, mbd_stream_t stream) {
    mbd::Epilogue ep;
    if (!fp8_epilogue(static_cast<int>(mode), &ep)) return MBD_ERR_INVALID_ARG;
    return norm_common(out_q, nullptr, ep, residual, x, weight, n_tokens, hidden, eps, scale,
                       reinterpret_cast<cudaStream_t>(stream));
}

mbd_status mbd_fused_add_rmsnorm_quant_nvfp4(uint8_t* out_q, uint8_t* out_sf, void* residual, const void* x,
                                             const void* weight, int64_t n_tokens, int64_t hidden, float eps,
                                             const float* tensor_scale, mbd_stream_t stream) {
    return norm_common(out_q, out_sf, mbd::kNvfp4, residual, x, weight, n_tokens, hidden, eps,
                       const_cast<float*>(tensor_scale), reinterpret_cast<cudaStream_t>(stream));
}

mbd_status mbd_fused_allreduce_add_rmsnorm(void* out, void* residual, const void* const* partials, int n_partials,
                                           const void* weight, int64_t n_tokens, int64_t hidden, float eps,
                                           mbd_stream_t stream) {
    if (n_partials < 1 || n_partials > MBD_MAX_PARTIALS || (n_tokens > 0 && !partials)) return MBD_ERR_INVALID_ARG;
    return norm_common(out, nullptr, mbd::kBf16, residual, nullptr, weight, n_tokens, hidden, eps, nullptr,
                       reinterpret_cast<cudaStream_t>(stream), partials, n_partials);
}

mbd_status mbd_fused_allreduce_add_rmsnorm_quant_fp8(uint8_t* out_q, void* residual, const void* const* partials,
                                                     int n_partials, const void* weight, int64_t n_tokens,
                                                     int64_t hidden, float eps, mbd_scale_mode mode, float* scale,
                                                     mbd_stream_t stream) {
    if (n_partials < 1 || n_partials > MBD_MAX_PARTIALS || (n_tokens > 0 && !partials)) return MBD_ERR_INVALID_ARG;
    mbd::Epilogue ep;
    if (!fp8_epilogue(static_cast<int>(mode), &ep)) return MBD_ERR_INVALID_ARG;
    return norm_common(out_q, nullptr, ep, residual, nullptr, weight, n_tokens, hidden, eps, scale,
                       reinterpret_cast<cudaStream_t>(stream), partials, n_partials);
}

mbd_status mbd_swiglu(void* out, const void* gate_up, int64_t n_tokens, int64_t inter, mbd_stream_t stream) {
    return swiglu_common(out, nullptr, mbd::kBf16, gate_up, n_tokens, inter, nullptr,
                         reinterpret_cast<cudaStream_t>(stream));
}

mbd_status mbd_swiglu_quant_fp8(uint8_t* out_q, const void* gate_up, int64_t n_tokens, int64_t inter,
                                mbd_scale_mode mode, float* scale, mbd_stream_t stream) {
    mbd::Epilogue ep;
    if (!fp8_epilogue(static_cast<int>(mode), &ep)) return MBD_ERR_INVALID_ARG;
    return swiglu_common(out_q, nullptr, ep, gate_up, n_tokens, inter, scale, reinterpret_cast<cudaStream_t>(stream));
}

mbd_status mbd_swiglu_quant_nvfp4(uint8_t* out_q, uint8_t* out_sf, const void* gate_up, int64_t n_tokens,
                                  int64_t inter, const float* tensor_scale, mbd_stream_t stream) {
    return swiglu_common(out_q, out_sf, mbd::kNvfp4, gate_up, n_tokens, inter, const_cast<float*>(tensor_scale),
                         reinterpret_cast<cudaStream_t>(stream));
}

mbd_status mbd_program_plan_build(const mbd_op* ops, int n_ops, mbd_program_plan* plan) {
    return build_program(ops, n_ops, reinterpret_cast<PlanImpl*>(plan));
}

mbd_status mbd_program_plan_launch(const mbd_program_plan* plan, mbd_stream_t stream) {
    return launch_plan(reinterpret_cast<const PlanImpl*>(plan), reinterpret_cast<cudaStream_t>(stream));
}

mbd_status mbd_tuning_set(const mbd_tuning_entry* entries, int n_entries) {
    if (n_entries < 0 || n_entries > MBD_MAX_TUNING_ENTRIES || (n_entries > 0 && !entries)) return MBD_ERR_INVALID_ARG;
    for (int i = 0; i < n_entries; ++i) {
        const mbd_tuning_entry& e = entries[i];
        const int v = e.vectors_per_thread;
        if (!valid_kind_mode(e.kind, e.mode) || e.reserved != 0 || e.tokens_min < 0 || e.tokens_max < e.tokens_min ||
            e.width_min < 0 || e.width_max < e.width_min || e.ctas_per_row < 1 || !(v == 1 || v == 2 || v == 4 || v == 8) ||
            e.threads < 32 || e.threads > 512 || e.threads % 32 != 0)
            return MBD_ERR_INVALID_ARG;
    }
    std::shared_ptr<const std::vector<mbd_tuning_entry>> t;
    if (n_entries > 0) t = std::make_shared<const std::vector<mbd_tuning_entry>>(entries, entries + n_entries);
    std::atomic_store(&g_tuning, t);
    return MBD_OK;
}

mbd_status mbd_launch_shape(int kind, int mode, int64_t n_tokens, int64_t width, int32_t* ctas_per_row,
                            int32_t* vectors_per_thread, int32_t* threads) {
    if (!valid_kind_mode(kind, mode) || n_tokens <= 0 || width <= 0 || !ctas_per_row || !vectors_per_thread || !threads)
        return MBD_ERR_INVALID_ARG;
    const bool norm = kind <= MBD_OP_ADD_RMSNORM_QUANT_NVFP4;
    const bool fp4 = kind == MBD_OP_ADD_RMSNORM_QUANT_NVFP4 || kind == MBD_OP_SWIGLU_QUANT_NVFP4;
    const bool dyn_swiglu = kind == MBD_OP_SWIGLU_QUANT_FP8 && mode == MBD_SCALE_DYNAMIC_PER_TOKEN;
    if (width % (fp4 ? 16 : 8) != 0) return MBD_ERR_MISALIGNED;
    if ((norm || dyn_swiglu) && width > MBD_MAX_REDUCED_WIDTH) return MBD_ERR_UNSUPPORTED;
    if (width > (int64_t{1} << 28)) return MBD_ERR_UNSUPPORTED;
    const int nvec = static_cast<int>(width / 8), sms = sm_count_of_current_device();
    mbd::RowPlan plan;
    if (!tuned_plan(kind, mode, n_tokens, width, nvec, norm || dyn_swiglu, fp4, sms, &plan) &&
        !plan_rows(n_tokens, nvec, norm ? Shape::kNorm : (dyn_swiglu ? Shape::kRowMax : Shape::kStream), sms, fp4, &plan))
        return MBD_ERR_UNSUPPORTED;
    if (dyn_swiglu) bulk_rule(n_tokens, nvec, sms, &plan);
    *ctas_per_row = plan.ctas_per_row;
    *vectors_per_thread = plan.vpt;
    *threads = plan.threads;
    return MBD_OK;
}

int mbd_tuning_get(mbd_tuning_entry* entries, int capacity) {
    const auto table = tuning_table();
    const int n = table ? static_cast<int>(table->size()) : 0;
    for (int i = 0; entries && i < n && i < capacity; ++i) entries[i] = (*table)[i];
    return n;
}

size_t mbd_program_schedule_bytes(void) { return kScheduleBytes; }

mbd_status mbd_program_plan_launch_static(const mbd_program_plan* plan, mbd_stream_t stream) {
    return launch_static(reinterpret_cast<const PlanImpl*>(plan), reinterpret_cast<cudaStream_t>(stream));
}

mbd_status mbd_program_plan_upload(const mbd_program_plan* plan, void* schedule, size_t schedule_bytes,
                                   mbd_stream_t stream) {
    return upload_plan(reinterpret_cast<const PlanImpl*>(plan), schedule, schedule_bytes,
                       reinterpret_cast<cudaStream_t>(stream));
}

mbd_status mbd_program_plan_launch_uploaded(const mbd_program_plan* plan, const void* schedule, mbd_stream_t stream) {
    return launch_uploaded(reinterpret_cast<const PlanImpl*>(plan), schedule, reinterpret_cast<cudaStream_t>(stream));
}

mbd_status mbd_run_independent(const mbd_op* ops, int n_ops, mbd_stream_t stream) {
    return run_independent(nullptr, nullptr, ops, n_ops, reinterpret_cast<cudaStream_t>(stream));
}

mbd_status mbd_run_independent_with_program(const mbd_program_plan* plan, const void* schedule, const mbd_op* ops,
                                            int n_ops, mbd_stream_t stream) {
    if (!plan) return MBD_ERR_INVALID_ARG;
    return run_independent(reinterpret_cast<const PlanImpl*>(plan), schedule, ops, n_ops,
                           reinterpret_cast<cudaStream_t>(stream));
}

mbd_status mbd_run_program(const mbd_op* ops, int n_ops, mbd_stream_t stream) {
    thread_local PlanImpl plan;   // about 14 KB: kept off the stack, reused by each call of this thread
    const mbd_status st = build_program(ops, n_ops, &plan);
    if (st != MBD_OK) return st;
    return launch_plan(&plan, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
