// rem_host.cu -- host side of the C ABI declared in include/rem.h.
//
// The contract it enforces is the one of mlx-native 0.18.0
// src/ops/row_exact_matvec.rs: `validate` (argument rules, output
// non-aliasing, buffer extents), `row_exact_reduction_nsg` and
// `RowExactMatvecSchedule::for_device` (a split factor that depends on the
// weight shape only, capped by what every kernel of the weight type can
// launch) and `dispatch_row_exact_matvec_scheduled` (refuse a launch above
// the kernels' thread limit instead of launching it).  Every rule is checked
// before anything is enqueued, so a rejected call writes nothing.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdlib>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "rem.h"
#include "rem_internal.h"

namespace rem {
namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

bool valid_wt(int wt) { return wt >= 0 && wt < kNumWt; }

const char* wt_name(int wt) {
    static const char* names[] = {"F16", "Q8_0", "Q4_K", "Q6_K", "Q5_0", "F32", "BF16", "A4G32", "A4G64",
                                  "A4G128", "A8G32", "A8G64", "A8G128"};
    return valid_wt(wt) ? names[wt] : "?";
}

uint64_t row_bytes_of(int wt, uint32_t k) {
    if (!valid_wt(wt)) return 0;
    return static_cast<uint64_t>(k / static_cast<uint32_t>(block_values(wt))) * block_bytes(wt);
}

uint32_t k_multiple(int wt) {
    if (is_affine(wt)) return static_cast<uint32_t>(affine_group(wt));
    switch (wt) {
    case kF16: case kF32: case kBF16: return 4;
    case kQ8_0: case kQ5_0: return 32;
    default: return 256;
    }
}

uint32_t w_align(int wt) {
    if (is_affine(wt)) return 4;  // 32-bit code words
    switch (wt) {
    case kF16: case kBF16: return 8;
    case kF32: return 4;
    case kQ4_K: return 16;  // 16-byte qs loads; 144-byte blocks keep it row to row
    default: return 2;
    }
}

uint32_t pow2_floor(uint64_t v) {
    uint32_t p = 1;
    while (static_cast<uint64_t>(p) * 2 <= v && p < (1u << 30)) p *= 2;
    return p;
}

// Last element index + 1 touched by a strided [batch, rows, cols] view.
uint64_t strided_extent(uint32_t batch, uint32_t bstride, uint32_t rows, uint32_t rstride, uint32_t cols) {
    return static_cast<uint64_t>(batch - 1) * bstride + static_cast<uint64_t>(rows - 1) * rstride + cols;
}

// REM_LOG_PLAN set in the environment: print each launch's schedule to stderr.
bool log_plans() {
    static const bool on = std::getenv("REM_LOG_PLAN") != nullptr;
    return on;
}

// REM_LAYOUT=0|1|2 in the environment: the lane layout every launch must use
// (read at each launch; -1 when unset or not one of those values).
int forced_layout() {
    const char* v = std::getenv("REM_LAYOUT");
    if (!v || v[0] < '0' || v[0] >= '0' + kNumLayouts || v[1] != '\0') return -1;
    return v[0] - '0';
}

// ---------------------------------------------------------------- driver entry points

using PFN_encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
using PFN_range = CUresult (*)(CUdeviceptr*, size_t*, CUdeviceptr);

struct Driver {
    PFN_encode encode = nullptr;
    PFN_range range = nullptr;
};

const Driver& driver() {
    static Driver d;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            d.encode = reinterpret_cast<PFN_encode>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            d.range = reinterpret_cast<PFN_range>(fn);
        cudaGetLastError();
    });
    return d;
}

// ---------------------------------------------------------------- per-device state

struct DeviceState {
    bool ready = false;
    int sms = 0;
    int smem_optin = 0;
    int smem_per_sm = 0;
    int max_threads[kNumWt][kMaxRows + 1][kNumLayouts] = {};  // per kernel <wt, m, layout>
};

std::mutex g_mu;
DeviceState g_dev[64];
std::map<std::tuple<const void*, int, int>, int> g_occ;  // (kernel, threads, smem) -> blocks per SM

int device_state(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return fail(REM_ECUDA, "rem_matvec: no current CUDA device");
    }
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& st = g_dev[dev];
    if (!st.ready) {
        if (cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&st.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&st.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
                cudaSuccess) {
            cudaGetLastError();
            return fail(REM_ECUDA, "rem_matvec: cannot query device %d", dev);
        }
        for (int wt = 0; wt < kNumWt; ++wt) {
            for (int m = 1; m <= kMaxRows; ++m)
                for (int l = 0; l < kNumLayouts; ++l) {
                    const void* fn = mv_kernel(wt, m, l);
                    if (!fn) continue;  // some layouts exist for some m only
                    cudaFuncAttributes fa;
                    if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess ||
                        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, st.smem_optin) !=
                            cudaSuccess) {
                        cudaGetLastError();
                        return fail(REM_ECUDA, "rem_matvec: cannot prepare the %s kernels on device %d (%s)",
                                    wt_name(wt), dev, "no sm_103a image for this device?");
                    }
                    st.max_threads[wt][m][l] = fa.maxThreadsPerBlock;
                }
        }
        st.ready = true;
    }
    *out = &st;
    return REM_OK;
}

int blocks_per_sm(const void* fn, int threads, int smem) {
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_tuple(fn, threads, smem);
    auto it = g_occ.find(key);
    if (it != g_occ.end()) return it->second;
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, threads, static_cast<size_t>(smem)) != cudaSuccess) {
        cudaGetLastError();
        nb = 0;
    }
    g_occ[key] = nb;
    return nb;
}

// Clusters of `split` blocks that can be resident at once (cached).
uint64_t resident_clusters(const void* fn, const cudaLaunchConfig_t& cfg, uint32_t split, int sms) {
    const int threads = static_cast<int>(cfg.blockDim.x);
    const int smem = static_cast<int>(cfg.dynamicSmemBytes);
    if (split <= 1) return static_cast<uint64_t>(blocks_per_sm(fn, threads, smem)) * sms;
    static std::map<std::tuple<const void*, int, int, uint32_t>, int> cache;
    std::lock_guard<std::mutex> lk(g_mu);
    const auto key = std::make_tuple(fn, threads, smem, split);
    auto it = cache.find(key);
    if (it != cache.end()) return static_cast<uint64_t>(it->second);
    cudaLaunchConfig_t c = cfg;
    c.gridDim = dim3(split * 64u);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &c) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    cache[key] = n;
    return static_cast<uint64_t>(n);
}

// A pointer the kernels may dereference, with at least `need` bytes after it
// when the allocation's extent is known.
int check_buffer(const void* p, uint64_t need, const char* what, int dev) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return fail(REM_EINVAL, "rem_matvec: %s (%p) is not a CUDA-visible pointer", what, p);
    }
    if (at.type == cudaMemoryTypeUnregistered)
        return fail(REM_EINVAL, "rem_matvec: %s (%p) is host memory not registered with CUDA", what, p);
    if (at.type == cudaMemoryTypeHost && at.devicePointer != p)
        return fail(REM_EINVAL, "rem_matvec: %s (%p) is pinned host memory; pass its device pointer", what, p);
    if (at.type == cudaMemoryTypeDevice && at.device != dev)
        return fail(REM_EINVAL, "rem_matvec: %s lives on device %d, the current device is %d", what, at.device, dev);
    if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) {
        const Driver& d = driver();
        if (d.range) {
            CUdeviceptr base = 0;
            size_t size = 0;
            if (d.range(&base, &size, reinterpret_cast<CUdeviceptr>(p)) == CUDA_SUCCESS) {
                const uint64_t avail = static_cast<uint64_t>(base) + size - reinterpret_cast<uint64_t>(p);
                if (avail < need)
                    return fail(REM_EINVAL, "rem_matvec: %s holds %llu bytes past the pointer, needs %llu", what,
                                static_cast<unsigned long long>(avail), static_cast<unsigned long long>(need));
            }
        }
    }
    return REM_OK;
}

struct Shape {
    uint32_t m, n, k, batch, xrs, xbs, yrs, ybs;
};

// The argument rules (validate), in the page's order.  Host-only: no CUDA call.
int validate_args(const void* W, int wt, const float* x, const float* y, const Shape& s, uint32_t split,
                  uint32_t rows_per_cta, bool any_m = false) {
    if (!valid_wt(wt)) return fail(REM_EINVAL, "rem_matvec: unknown weight type %d", wt);
    if (s.m == 0 || (!any_m && s.m > kMaxRows))
        return fail(REM_EINVAL, any_m ? "rem_matvec_many: m (%u) must be >= 1" : "rem_matvec: m (%u) must be in 1..=8",
                    s.m);
    if (s.n == 0 || s.k == 0 || s.batch == 0)
        return fail(REM_EINVAL, "rem_matvec: n (%u), k (%u) and batch (%u) must be > 0", s.n, s.k, s.batch);
    if (split > REM_MAX_SPLIT)
        return fail(REM_EINVAL, "rem_matvec: split (%u) must be 0 (auto) or in 1..=%d", split, REM_MAX_SPLIT);
    if (!(rows_per_cta == 0 || rows_per_cta == 32 || rows_per_cta == 64 || rows_per_cta == 128))
        return fail(REM_EINVAL, "rem_matvec: rows_per_cta (%u) must be 0, 32, 64 or 128", rows_per_cta);
    if (!W || !x || !y) return fail(REM_EINVAL, "rem_matvec: W, x and y must be non-null");
    if (s.k % k_multiple(wt) != 0)
        return fail(REM_EINVAL, "rem_matvec: k (%u) must be a multiple of %u for %s", s.k, k_multiple(wt),
                    wt_name(wt));
    if (s.xrs % 4 != 0 || s.xbs % 4 != 0 || reinterpret_cast<uintptr_t>(x) % 16 != 0)
        return fail(REM_EINVAL,
                    "rem_matvec: input strides (%u, %u) must be multiples of 4 and the input pointer 16-byte aligned",
                    s.xrs, s.xbs);
    if (reinterpret_cast<uintptr_t>(W) % w_align(wt) != 0 || reinterpret_cast<uintptr_t>(y) % 4 != 0)
        return fail(REM_EINVAL, "rem_matvec: weight pointer must be %u-byte and output pointer 4-byte aligned",
                    w_align(wt));
    // Output elements must not alias: rows of one product and the products of
    // one call write disjoint ranges (either layout order is accepted).
    const bool rows_disjoint = s.m == 1 || s.yrs >= s.n;
    bool disjoint;
    if (s.batch == 1) {
        disjoint = rows_disjoint;
    } else if (s.m == 1) {
        disjoint = s.ybs >= s.n;
    } else if (s.yrs >= s.ybs) {
        disjoint = s.ybs >= s.n &&
                   static_cast<uint64_t>(s.yrs) >= static_cast<uint64_t>(s.batch - 1) * s.ybs + s.n;
    } else {
        disjoint = rows_disjoint && static_cast<uint64_t>(s.ybs) >= static_cast<uint64_t>(s.m - 1) * s.yrs + s.n;
    }
    if (!disjoint)
        return fail(REM_EINVAL,
                    "rem_matvec: output strides overlap: y_row_stride %u, y_batch_stride %u, m %u, n %u, batch %u",
                    s.yrs, s.ybs, s.m, s.n, s.batch);
    if (static_cast<uint64_t>(s.m - 1) * s.yrs + s.n > 0xFFFFFFFFull)
        return fail(REM_EINVAL, "rem_matvec: output row extent exceeds u32");
    return REM_OK;
}

uint32_t auto_split(int wt, uint64_t rows, uint32_t k) {
    const uint64_t nchunk = (k + chunk_values(wt) - 1) / chunk_values(wt);
    const uint64_t groups = (rows + kLanes - 1) / kLanes;
    const uint64_t per = groups >= 2048 ? 1 : 2048 / groups;
    uint32_t s = pow2_floor(per);
    if (s > static_cast<uint32_t>(kMaxSplit)) s = kMaxSplit;
    const uint32_t cmax = pow2_floor(nchunk == 0 ? 1 : nchunk);
    return s < cmax ? s : cmax;
}

// Planner weight of a lane layout.  Four rows per lane (two of them in each
// of two lane groups) share every input load four ways (2.0; they exist only
// where they measured faster).  Two rows per lane in one group share
// every input load (1.8x; 1.3x at m = 1, where the input loads weigh less
// against the decode, except for affine weights, whose per-group scale loads
// the second row of each lane overlaps).  Two lane groups (H = 2) share input
// loads too but stage and decode each weight row twice, which pays off from
// four input rows up, or at any m for weights without a per-block decode
// (F16, BF16, F32) and for affine weights.
double layout_weight(int wt, int m, int nr0, int h) {
    if (nr0 == 2 && h == 2) return 2.0;  // F16 / BF16 at m = 6, 8 (the only kernels of this layout)
    if (nr0 == 2) return (m >= 2 || is_affine(wt)) ? 1.8 : 1.3;
    if (h == 1) return 1.0;
    const bool cheap = wt == kF16 || wt == kBF16 || wt == kF32 || is_affine(wt);
    return (m >= 4 || cheap) ? 1.2 : 0.9;
}

struct Plan {
    int nr0, h, warps, stages, smem;
    uint32_t cpb, grid;
    bool aligned, pdl;
};

// Optional epilogue of a launch: y = alpha * acc + beta * c.
struct Epilogue {
    uint32_t mode = 0;  // 0 none, 1 alpha only, 2 alpha and beta * c
    float alpha = 1.0f, beta = 0.0f;
    const float* c = nullptr;
    uint32_t crs = 0, cbs = 0;
};

// Scale and bias arrays of an affine weight (binary16, one per group and row).
struct AffineArgs {
    const uint16_t* scales = nullptr;
    const uint16_t* biases = nullptr;
};

int launch_matvec(const void* W, int wt, const float* x, float* y, const Shape& s, uint32_t split,
                  uint32_t rows_per_cta, void* stream, const Epilogue& epi = Epilogue(),
                  const AffineArgs* aff = nullptr) {
    int rc = validate_args(W, wt, x, y, s, split, rows_per_cta);
    if (rc != REM_OK) return rc;
    if (is_affine(wt) && !aff)
        return fail(REM_EINVAL, "rem_matvec: %s weights need their scales and biases: use rem_matvec_affine",
                    wt_name(wt));
    if (!is_affine(wt) && aff) return fail(REM_EINVAL, "rem_matvec_affine: %s is not an affine type", wt_name(wt));
    const uint64_t rb = row_bytes_of(wt, s.k);
    const uint64_t rows = static_cast<uint64_t>(s.batch) * s.n;
    DeviceState* ds = nullptr;
    if ((rc = device_state(&ds)) != REM_OK) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    if ((rc = check_buffer(W, rb * rows, "weight", dev)) != REM_OK) return rc;
    if ((rc = check_buffer(x, 4 * strided_extent(s.batch, s.xbs, s.m, s.xrs, s.k), "input", dev)) != REM_OK)
        return rc;
    if ((rc = check_buffer(y, 4 * strided_extent(s.batch, s.ybs, s.m, s.yrs, s.n), "output", dev)) != REM_OK)
        return rc;
    if (aff) {
        const uint64_t sb = 2 * rows * (s.k / static_cast<uint32_t>(affine_group(wt)));
        if (!aff->scales || !aff->biases || reinterpret_cast<uintptr_t>(aff->scales) % 2 != 0 ||
            reinterpret_cast<uintptr_t>(aff->biases) % 2 != 0)
            return fail(REM_EINVAL, "rem_matvec_affine: scales and biases must be non-null and 2-byte aligned");
        if ((rc = check_buffer(aff->scales, sb, "scales", dev)) != REM_OK) return rc;
        if ((rc = check_buffer(aff->biases, sb, "biases", dev)) != REM_OK) return rc;
    }

    // split = CTAs per cluster that share one row group's K ranges
    uint32_t S = split ? split : auto_split(wt, rows, s.k);
    if (!split && S > static_cast<uint32_t>(kMaxSplit)) S = kMaxSplit;
    if (S > static_cast<uint32_t>(kMaxSplit))
        return fail(REM_ELAUNCH,
                    "rem_matvec: split %u needs clusters of %u thread blocks but the %s kernels launch clusters of "
                    "at most %d",
                    S, S, wt_name(wt), kMaxSplit);
    const uint32_t nchunk = (s.k + chunk_values(wt) - 1) / chunk_values(wt);

    Plan p{};
    // TMA staging needs 16-byte aligned rows and encodable tensor maps.
    // Inputs: [batch][m][k] f32 with the caller's strides, dimensions ordered
    // by increasing stride; either order stages the box as [m][chunk].
    alignas(64) CUtensorMap wmap, xmap;
    bool x_bm = false;
    std::memset(&wmap, 0, sizeof(wmap));
    std::memset(&xmap, 0, sizeof(xmap));
    p.aligned = reinterpret_cast<uintptr_t>(W) % 16 == 0 && rb % 16 == 0 && rows < (1ull << 31) &&
                rb / 2 < (1ull << 32) && driver().encode != nullptr;
    if (p.aligned) {
        const uint64_t xrs = s.m == 1 ? s.k : s.xrs;
        const uint64_t xbs = s.batch == 1 ? xrs * s.m : s.xbs;
        x_bm = xbs < xrs;
        const cuuint64_t gdim[3] = {s.k, x_bm ? s.batch : s.m, x_bm ? s.m : s.batch};
        const cuuint64_t gstride[2] = {4 * (x_bm ? xbs : xrs), 4 * (x_bm ? xrs : xbs)};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(chunk_values(wt)), x_bm ? 1u : s.m, x_bm ? s.m : 1u};
        const cuuint32_t estride[3] = {1, 1, 1};
        p.aligned = xrs > 0 && xbs > 0 &&
                    driver().encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(x), gdim,
                                    gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }

    // Lane layout (NR0 rows per lane and H lane groups), row-block width G
    // (consumer warps per CTA) and ring depth D: the fitting combination with
    // the best score.  The score models a kernel that is bound by how many
    // consumer warps each SM keeps busy (latency of shared-memory loads and
    // stage waits): the average consumer warps per SM (saturating at 8), times
    // the lane layout's weight (layout_weight), a single stage (no copy /
    // compute overlap) 0.7x, the producer warp's share (G/(G+1))^2, 20% less
    // per stage beyond two (deeper rings cost residency for no gain), all
    // scaled by the share of resident CTA slots the last wave of row blocks
    // keeps busy.  The weights were fitted to timings of every (layout, G, D)
    // on GB300 for the five formats at 4096..128256 rows.
    cudaLaunchConfig_t cfg{};
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    if (S > 1) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
        attr[cfg.numAttrs].val.clusterDim.x = S;
        attr[cfg.numAttrs].val.clusterDim.y = 1;
        attr[cfg.numAttrs].val.clusterDim.z = 1;
        ++cfg.numAttrs;
    }
    double best = -1.0;
    const void* fn = nullptr;
    int last_cap = 0;
    const int pinned = forced_layout();
    for (int l = kNumLayouts - 1; l >= 0; --l) {
        const void* f = mv_kernel(wt, static_cast<int>(s.m), l);
        if (!f || (pinned >= 0 && l != pinned)) continue;
        const int nr0 = layout_nr0(l), h = layout_h(l);
        const uint32_t rpw = static_cast<uint32_t>(kLanes * nr0);
        const int cap = ds->max_threads[wt][s.m][l];
        for (int g = kMaxWarps; g >= 1; g /= 2) {
            if (rows_per_cta ? static_cast<uint32_t>(g) * rpw != rows_per_cta
                             : (g > 4 || static_cast<uint32_t>(g) * rpw > 256u))
                continue;
            if ((g + 1) * 32 > cap) {
                last_cap = cap;
                continue;
            }
            const uint64_t nb = static_cast<uint64_t>(s.batch) * ((s.n + rpw * g - 1) / (rpw * g));
            const uint64_t units = nb * S;
            const uint64_t per_cta = ((nchunk + S - 1) / S) * ((units + 2ull * ds->sms - 1) / (2ull * ds->sms));
            const int dmax = static_cast<int>(std::min<uint64_t>(kMaxStages, std::max<uint64_t>(2, per_cta)));
            for (int d = 1; d <= dmax; ++d) {
                const int sm = static_cast<int>(mv_smem_bytes(wt, nr0, h, g, d, static_cast<int>(s.m), S));
                if (sm > ds->smem_optin) continue;
                cfg.blockDim = dim3(static_cast<unsigned>((g + 1) * 32));
                cfg.dynamicSmemBytes = static_cast<size_t>(sm);
                const uint64_t slots = resident_clusters(f, cfg, S, ds->sms) * S;
                if (slots == 0) continue;
                const uint64_t ctas = std::min(units, slots);
                const uint64_t waves = (units + ctas - 1) / ctas;
                const double eff = static_cast<double>(units) / static_cast<double>(waves * ctas);
                const double warps_sm = static_cast<double>(ctas) / ds->sms * g;
                const double gf = static_cast<double>(g) / (g + 1);
                double score = std::min(warps_sm, 8.0) * layout_weight(wt, static_cast<int>(s.m), nr0, h) *
                               (d == 1 ? 0.7 : 1.0) * gf * gf *
                               (1.0 - 0.2 * std::max(0, d - 2)) * eff;
                if (score > best) {
                    best = score;
                    fn = f;
                    p.nr0 = nr0;
                    p.h = h;
                    p.warps = g;
                    p.stages = d;
                    p.smem = sm;
                }
            }
        }
    }
    if (best < 0) {
        if (pinned >= 0 && !mv_kernel(wt, static_cast<int>(s.m), pinned))
            return fail(REM_ELAUNCH, "rem_matvec: lane layout %d (REM_LAYOUT) has no %s kernel for m = %u", pinned,
                        wt_name(wt), s.m);
        if (last_cap)
            return fail(REM_ELAUNCH, "rem_matvec: %u rows per block exceed the %s kernel's limit of %d threads",
                        rows_per_cta, wt_name(wt), last_cap);
        return fail(REM_ELAUNCH, "rem_matvec: no %s row block fits the device's shared memory", wt_name(wt));
    }
    const uint32_t rows_per_warp = static_cast<uint32_t>(kLanes * p.nr0);
    p.cpb = (s.n + rows_per_warp * p.warps - 1) / (rows_per_warp * p.warps);
    const uint64_t nblocks = static_cast<uint64_t>(p.cpb) * s.batch;
    if (nblocks > 0x7FFFFFFFull)
        return fail(REM_EINVAL, "rem_matvec: too many row blocks (%llu)", static_cast<unsigned long long>(nblocks));
    const int threads = (p.warps + 1) * 32;
    if (p.aligned) {
        // weights as [rows][row_bytes/2] u16, one box = the row block's rows x one chunk
        const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(rb / 2), static_cast<cuuint64_t>(rows)};
        const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(rb)};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(chunk_box(wt) / 2), rows_per_warp * p.warps};
        const cuuint32_t estride[2] = {1, 1};
        p.aligned = driver().encode(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(W), gdim, gstride,
                                    box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }

    // persistent grid: as many clusters as can be resident, at most one per row block
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(p.smem);
    const uint64_t resident = resident_clusters(fn, cfg, S, ds->sms);
    if (resident == 0)
        return fail(REM_ELAUNCH, "rem_matvec: a cluster of %u blocks of %d threads and %d bytes does not fit",
                    S, threads, p.smem);
    const uint64_t ncl = std::min<uint64_t>(nblocks, resident);
    // When fewer CTAs run than can be resident, the block scheduler fills SMs
    // to their occupancy limit and leaves others idle.  Asking for more
    // (unused) shared memory per CTA caps the CTAs per SM at the even share,
    // ceil(ctas / SMs), which spreads the grid over the SMs -- kept only if
    // the whole grid still fits at once.
    if (ncl < resident) {
        const uint64_t per_sm = (ncl * S + ds->sms - 1) / ds->sms;
        const int cap = static_cast<int>(std::min<uint64_t>(static_cast<uint64_t>(ds->smem_optin),
                                                            static_cast<uint64_t>(ds->smem_per_sm) / per_sm - 1024));
        if (cap > p.smem && blocks_per_sm(fn, threads, p.smem) > static_cast<int>(per_sm)) {
            cfg.dynamicSmemBytes = static_cast<size_t>(cap);
            if (resident_clusters(fn, cfg, S, ds->sms) >= ncl) p.smem = cap;
            cfg.dynamicSmemBytes = static_cast<size_t>(p.smem);
        }
    }
    p.grid = static_cast<uint32_t>(ncl * S);
    cfg.gridDim = dim3(p.grid);
    // Programmatic dependent launch: the kernel may start while the previous
    // kernel of the stream finishes (it waits for it, griddepcontrol.wait,
    // before reading x or W into shared memory and before writing y), and
    // prefetches its first weights into L2 meanwhile.  That pays where the
    // launch is short next to its start-up latency -- from m = 4 up (compute
    // bound) below 256 MB of weights, at any m below 24 MB -- and costs
    // throughput on long bandwidth-bound launches, which keep plain stream
    // order.  Scheduling only: the arithmetic is the same either way.
    const uint64_t wbytes = rb * rows;
    p.pdl = (s.m >= 4 && wbytes <= (256ull << 20)) || wbytes <= (24ull << 20);
    if (p.pdl) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
        ++cfg.numAttrs;
    }
    if (log_plans())
        fprintf(stderr,
                "rem_matvec plan: %s m %u n %u k %u batch %u split %u nr0 %d h %d warps %d stages %d smem %d grid %u "
                "row_blocks %llu tma %d pdl %d\n",
                wt_name(wt), s.m, s.n, s.k, s.batch, S, p.nr0, p.h, p.warps, p.stages, p.smem, p.grid,
                static_cast<unsigned long long>(nblocks), static_cast<int>(p.aligned), static_cast<int>(p.pdl));

    MvArgs a{};
    a.w = static_cast<const uint8_t*>(W);
    a.x = x;
    a.y = y;
    a.row_bytes = rb;
    a.n = s.n;
    a.k = s.k;
    a.xrs = s.xrs;
    a.xbs = s.xbs;
    a.yrs = s.yrs;
    a.ybs = s.ybs;
    a.split = S;
    a.nchunk = nchunk;
    a.cpb = p.cpb;
    a.batch = s.batch;
    a.stages = static_cast<uint32_t>(p.stages);
    a.aligned = p.aligned ? 1u : 0u;
    a.x_bm = x_bm ? 1u : 0u;
    a.pdl = p.pdl ? 1u : 0u;
    a.epi = epi.mode;
    a.alpha = epi.alpha;
    a.beta = epi.beta;
    a.c = epi.c;
    a.crs = epi.crs;
    a.cbs = epi.cbs;
    if (aff) {
        a.scales = aff->scales;
        a.biases = aff->biases;
        a.ngroups = s.k / static_cast<uint32_t>(affine_group(wt));
    }

    void* args[3] = {&wmap, &xmap, &a};
    const cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(REM_ECUDA, "rem_matvec: launch failed: %s", cudaGetErrorString(e));
    }
    return REM_OK;
}

int check_rows_buffer(const void* W, int wt, uint32_t rows, uint32_t k, const char* fn_name) {
    if (!valid_wt(wt)) return fail(REM_EINVAL, "%s: unknown weight type %d", fn_name, wt);
    if (rows == 0 || k == 0) return fail(REM_EINVAL, "%s: rows (%u) and k (%u) must be > 0", fn_name, rows, k);
    if (k % k_multiple(wt) != 0)
        return fail(REM_EINVAL, "%s: k (%u) must be a multiple of %u for %s", fn_name, k, k_multiple(wt),
                    wt_name(wt));
    if (!W) return fail(REM_EINVAL, "%s: null weight pointer", fn_name);
    if (reinterpret_cast<uintptr_t>(W) % w_align(wt) != 0)
        return fail(REM_EINVAL, "%s: weight pointer must be %u-byte aligned", fn_name, w_align(wt));
    return REM_OK;
}

}  // namespace

const void* mv_kernel(int wt, int m, int layout) {
    const bool lo = m <= 4;
    switch (wt) {
    case kF16: return lo ? mv_kernel_f16_a(m, layout) : mv_kernel_f16_b(m, layout);
    case kQ8_0: return lo ? mv_kernel_q8_0_a(m, layout) : mv_kernel_q8_0_b(m, layout);
    case kQ5_0: return lo ? mv_kernel_q5_0_a(m, layout) : mv_kernel_q5_0_b(m, layout);
    case kQ4_K: return lo ? mv_kernel_q4_k_a(m, layout) : mv_kernel_q4_k_b(m, layout);
    case kQ6_K: return lo ? mv_kernel_q6_k_a(m, layout) : mv_kernel_q6_k_b(m, layout);
    case kF32: return lo ? mv_kernel_f32_a(m, layout) : mv_kernel_f32_b(m, layout);
    case kBF16: return lo ? mv_kernel_bf16_a(m, layout) : mv_kernel_bf16_b(m, layout);
    case kA4G32: return lo ? mv_kernel_a4g32_a(m, layout) : mv_kernel_a4g32_b(m, layout);
    case kA4G64: return lo ? mv_kernel_a4g64_a(m, layout) : mv_kernel_a4g64_b(m, layout);
    case kA4G128: return lo ? mv_kernel_a4g128_a(m, layout) : mv_kernel_a4g128_b(m, layout);
    case kA8G32: return lo ? mv_kernel_a8g32_a(m, layout) : mv_kernel_a8g32_b(m, layout);
    case kA8G64: return lo ? mv_kernel_a8g64_a(m, layout) : mv_kernel_a8g64_b(m, layout);
    case kA8G128: return lo ? mv_kernel_a8g128_a(m, layout) : mv_kernel_a8g128_b(m, layout);
    default: return nullptr;
    }
}

}  // namespace rem

using namespace rem;

extern "C" {

int rem_matvec(const void* W, int wtype, uint32_t n, uint32_t k, uint32_t batch, const float* x, uint32_t m,
               uint32_t x_batch_stride, float* y, uint32_t y_batch_stride, void* stream) {
    g_err[0] = '\0';
    Shape s{m, n, k, batch, k, x_batch_stride, n, y_batch_stride};
    if (batch > 1 && static_cast<uint64_t>(x_batch_stride) < static_cast<uint64_t>(m) * k) {
        // token-major grouped projection: x [m, batch*k], y [m, batch*n]
        const uint64_t xrs = static_cast<uint64_t>(batch) * k, yrs = static_cast<uint64_t>(batch) * n;
        if (xrs > 0xFFFFFFFFull || yrs > 0xFFFFFFFFull)
            return fail(REM_EINVAL, "rem_matvec: inferred token-major row stride exceeds u32; use rem_matvec_ex");
        s.xrs = static_cast<uint32_t>(xrs);
        s.yrs = static_cast<uint32_t>(yrs);
    }
    return launch_matvec(W, wtype, x, y, s, 0, 0, stream);
}

int rem_matvec_ex(const void* W, int wtype, uint32_t n, uint32_t k, uint32_t batch, const float* x, uint32_t m,
                  uint32_t x_row_stride, uint32_t x_batch_stride, float* y, uint32_t y_row_stride,
                  uint32_t y_batch_stride, uint32_t split, uint32_t rows_per_cta, void* stream) {
    g_err[0] = '\0';
    const Shape s{m, n, k, batch, x_row_stride, x_batch_stride, y_row_stride, y_batch_stride};
    return launch_matvec(W, wtype, x, y, s, split, rows_per_cta, stream);
}

int rem_matvec_axpby(const void* W, int wtype, uint32_t n, uint32_t k, uint32_t batch, const float* x, uint32_t m,
                     uint32_t x_row_stride, uint32_t x_batch_stride, float* y, uint32_t y_row_stride,
                     uint32_t y_batch_stride, float alpha, float beta, const float* c, uint32_t c_row_stride,
                     uint32_t c_batch_stride, void* stream) {
    g_err[0] = '\0';
    const Shape s{m, n, k, batch, x_row_stride, x_batch_stride, y_row_stride, y_batch_stride};
    Epilogue e;
    e.alpha = alpha;
    e.beta = beta;
    if (beta != 0.0f) {
        if (!c || reinterpret_cast<uintptr_t>(c) % 4 != 0)
            return fail(REM_EINVAL, "rem_matvec: c must be non-null and 4-byte aligned when beta != 0");
        // c may be y itself (same strides: each element is read, then written, by one thread);
        // any other overlap between c and y is refused
        const uint64_t cext = 4 * strided_extent(batch, c_batch_stride, m, c_row_stride, n);
        const uint64_t yext = 4 * strided_extent(batch, y_batch_stride, m, y_row_stride, n);
        const uintptr_t c0 = reinterpret_cast<uintptr_t>(c), y0 = reinterpret_cast<uintptr_t>(y);
        const bool same = c0 == y0 && c_row_stride == y_row_stride && c_batch_stride == y_batch_stride;
        if (!same && c0 < y0 + yext && y0 < c0 + cext)
            return fail(REM_EINVAL, "rem_matvec: c overlaps y (only c == y with the same strides is allowed)");
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) {
            cudaGetLastError();
            return fail(REM_ECUDA, "rem_matvec: no current CUDA device");
        }
        int rc = validate_args(W, wtype, x, y, s, 0, 0);
        if (rc != REM_OK) return rc;
        if ((rc = check_buffer(c, cext, "addend c", dev)) != REM_OK) return rc;
        e.mode = 2;
        e.c = c;
        e.crs = c_row_stride;
        e.cbs = c_batch_stride;
    } else if (alpha != 1.0f) {
        e.mode = 1;
    }
    return launch_matvec(W, wtype, x, y, s, 0, 0, stream, e);
}

int rem_matvec_affine(const void* codes, const uint16_t* scales, const uint16_t* biases, int wtype, uint32_t n,
                      uint32_t k, uint32_t batch, const float* x, uint32_t m, uint32_t x_row_stride,
                      uint32_t x_batch_stride, float* y, uint32_t y_row_stride, uint32_t y_batch_stride,
                      uint32_t split, void* stream) {
    g_err[0] = '\0';
    if (!is_affine(wtype)) return fail(REM_EINVAL, "rem_matvec_affine: %d is not an affine weight type", wtype);
    if (!scales || !biases)
        return fail(REM_EINVAL, "rem_matvec_affine: scales and biases must be non-null and 2-byte aligned");
    const Shape s{m, n, k, batch, x_row_stride, x_batch_stride, y_row_stride, y_batch_stride};
    AffineArgs aff;
    aff.scales = scales;
    aff.biases = biases;
    return launch_matvec(codes, wtype, x, y, s, split, 0, stream, Epilogue(), &aff);
}

int rem_dequantize_affine(const void* codes, const uint16_t* scales, const uint16_t* biases, int wtype,
                          uint32_t rows, uint32_t k, float* out, void* stream) {
    g_err[0] = '\0';
    if (!is_affine(wtype)) return fail(REM_EINVAL, "rem_dequantize_affine: %d is not an affine weight type", wtype);
    int rc = check_rows_buffer(codes, wtype, rows, k, "rem_dequantize_affine");
    if (rc != REM_OK) return rc;
    if (!scales || !biases || reinterpret_cast<uintptr_t>(scales) % 2 || reinterpret_cast<uintptr_t>(biases) % 2)
        return fail(REM_EINVAL, "rem_dequantize_affine: scales and biases must be non-null and 2-byte aligned");
    if (!out || reinterpret_cast<uintptr_t>(out) % 4 != 0)
        return fail(REM_EINVAL, "rem_dequantize_affine: output must be non-null and 4-byte aligned");
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return fail(REM_ECUDA, "rem_dequantize_affine: no current CUDA device");
    }
    const uint64_t sb = 2ull * rows * (k / static_cast<uint32_t>(affine_group(wtype)));
    if ((rc = check_buffer(codes, row_bytes_of(wtype, k) * rows, "codes", dev)) != REM_OK) return rc;
    if ((rc = check_buffer(scales, sb, "scales", dev)) != REM_OK) return rc;
    if ((rc = check_buffer(biases, sb, "biases", dev)) != REM_OK) return rc;
    if ((rc = check_buffer(out, 4ull * rows * k, "output", dev)) != REM_OK) return rc;
    if (launch_dequantize_affine(static_cast<const uint32_t*>(codes), scales, biases, wtype, rows, k, out, stream) !=
        0)
        return fail(REM_ECUDA, "rem_dequantize_affine: launch failed");
    return REM_OK;
}

int rem_matvec_many(const void* W, int wtype, uint32_t n, uint32_t k, uint32_t batch, const float* x, uint32_t m,
                    uint32_t x_row_stride, uint32_t x_batch_stride, float* y, uint32_t y_row_stride,
                    uint32_t y_batch_stride, uint32_t split, void* stream) {
    g_err[0] = '\0';
    const Shape all{m, n, k, batch, x_row_stride, x_batch_stride, y_row_stride, y_batch_stride};
    // every rule for the whole call (output aliasing over all m rows
    // included) and every group's rules are checked before the first launch
    int rc = validate_args(W, wtype, x, y, all, split, 0, true);
    if (rc != REM_OK) return rc;
    for (uint32_t j0 = 0; j0 < m; j0 += kMaxRows) {
        const Shape g{std::min<uint32_t>(kMaxRows, m - j0), n, k, batch, x_row_stride, x_batch_stride,
                      y_row_stride, y_batch_stride};
        if ((rc = validate_args(W, wtype, x + static_cast<uint64_t>(j0) * x_row_stride, y +
                                static_cast<uint64_t>(j0) * y_row_stride, g, split, 0)) != REM_OK)
            return rc;
    }
    // the split comes from the shape, so every group (and an m = 1 call)
    // uses the same one
    const uint32_t S = split ? split : auto_split(wtype, static_cast<uint64_t>(batch) * n, k);
    for (uint32_t j0 = 0; j0 < m; j0 += kMaxRows) {
        const Shape g{std::min<uint32_t>(kMaxRows, m - j0), n, k, batch, x_row_stride, x_batch_stride,
                      y_row_stride, y_batch_stride};
        rc = launch_matvec(W, wtype, x + static_cast<uint64_t>(j0) * x_row_stride,
                           y + static_cast<uint64_t>(j0) * y_row_stride, g, S, 0, stream);
        if (rc != REM_OK) return rc;
    }
    return REM_OK;
}

uint64_t rem_row_bytes(int wtype, uint32_t k) { return row_bytes_of(wtype, k); }

uint32_t rem_split_factor(int wtype, uint32_t rows, uint32_t k) {
    if (!valid_wt(wtype) || rows == 0 || k == 0) return 0;
    g_err[0] = '\0';
    return auto_split(wtype, rows, k);
}

int rem_dequantize(const void* W, int wtype, uint32_t rows, uint32_t k, float* out, void* stream) {
    g_err[0] = '\0';
    if (is_affine(wtype)) return fail(REM_EINVAL, "rem_dequantize: use rem_dequantize_affine for affine weights");
    int rc = check_rows_buffer(W, wtype, rows, k, "rem_dequantize");
    if (rc != REM_OK) return rc;
    if (!out || reinterpret_cast<uintptr_t>(out) % 4 != 0)
        return fail(REM_EINVAL, "rem_dequantize: output must be non-null and 4-byte aligned");
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return fail(REM_ECUDA, "rem_dequantize: no current CUDA device");
    }
    const uint64_t rb = row_bytes_of(wtype, k);
    if ((rc = check_buffer(W, rb * rows, "weight", dev)) != REM_OK) return rc;
    if ((rc = check_buffer(out, 4ull * rows * k, "output", dev)) != REM_OK) return rc;
    if (launch_dequantize(static_cast<const uint8_t*>(W), wtype, rows, k, rb, out, stream) != 0)
        return fail(REM_ECUDA, "rem_dequantize: launch failed");
    return REM_OK;
}

int rem_quantize(const float* src, int wtype, uint32_t rows, uint32_t k, void* W, void* stream) {
    g_err[0] = '\0';
    if (is_affine(wtype)) return fail(REM_EINVAL, "rem_quantize: affine weights are not produced here");
    int rc = check_rows_buffer(W, wtype, rows, k, "rem_quantize");
    if (rc != REM_OK) return rc;
    if (!src || reinterpret_cast<uintptr_t>(src) % 4 != 0)
        return fail(REM_EINVAL, "rem_quantize: input must be non-null and 4-byte aligned");
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return fail(REM_ECUDA, "rem_quantize: no current CUDA device");
    }
    const uint64_t rb = row_bytes_of(wtype, k);
    if ((rc = check_buffer(src, 4ull * rows * k, "input", dev)) != REM_OK) return rc;
    if ((rc = check_buffer(W, rb * rows, "weight", dev)) != REM_OK) return rc;
    if (launch_quantize(src, wtype, rows, k, rb, static_cast<uint8_t*>(W), stream) != 0)
        return fail(REM_ECUDA, "rem_quantize: launch failed");
    return REM_OK;
}

const char* rem_last_error(void) { return g_err; }

int rem_version(void) { return 1; }

}  // extern "C"
