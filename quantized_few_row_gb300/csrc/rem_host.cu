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
    static const char* names[] = {"F16",   "Q8_0",  "Q4_K",  "Q6_K",   "Q5_0",  "F32",   "BF16",  "A4G32",
                                  "A4G64", "A4G128", "A8G32", "A8G64", "A8G128", "A3G32", "A3G64", "A3G128",
                                  "A5G32", "A5G64",  "A5G128", "A6G32", "A6G64", "A6G128"};
    static_assert(sizeof(names) / sizeof(names[0]) == kNumWt, "one name per weight type");
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

// Description of the calling thread's last launch (rem_last_plan).
thread_local char g_plan[256] = "";


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

// The status word every launch reports a timed-out wait into (one per device:
// the module's __device__ variable exists once on every device that loads
// the library).
__device__ uint32_t g_status_word;

struct DeviceState {
    bool ready = false;
    int sms = 0;
    int smem_optin = 0;
    int smem_per_sm = 0;
    uint32_t* status = nullptr;  // device address of g_status_word on this device
    int max_threads[kNumWt][kMaxRows + 1][kNumLayouts] = {};  // per kernel <wt, m, layout>
};

std::mutex g_mu;
DeviceState g_dev[64];
// (device, kernel, threads, smem, split) -> resident thread blocks per SM (split 1) or clusters per device
std::map<std::tuple<int, const void*, int, int, uint32_t>, int> g_occ;

int device_state(DeviceState** out, int* dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return fail(REM_ECUDA, "rem_matvec: no current CUDA device");
    }
    *dev_out = dev;
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
        void* sp = nullptr;
        if (cudaGetSymbolAddress(&sp, g_status_word) != cudaSuccess || !sp) {
            cudaGetLastError();
            return fail(REM_ECUDA, "rem_matvec: no status word on device %d (no sm_103a image for this device?)",
                        dev);
        }
        st.status = static_cast<uint32_t*>(sp);
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
            if (tc_format(wt))
                for (int mp = 1; mp <= tc_max_mp(wt); mp *= 2)
                    for (int cm = 0; cm < 2; ++cm) {
                    const void* fn = tc_kernel(wt, mp, cm != 0);
                    if (!fn) continue;  // not every width takes both conversion modes
                    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                    st.smem_optin) != cudaSuccess) {
                        cudaGetLastError();
                        return fail(REM_ECUDA, "rem_matvec: cannot prepare the %s tensor-core kernels on device %d",
                                    wt_name(wt), dev);
                    }
                }
        }
        st.ready = true;
    }
    *out = &st;
    return REM_OK;
}

// Resident thread blocks per SM (split <= 1) or resident clusters of `split`
// blocks on the device, for a kernel, block size and dynamic shared memory
// (cached per device).
uint64_t resident(int dev, const void* fn, const cudaLaunchConfig_t& cfg, uint32_t split) {
    const int threads = static_cast<int>(cfg.blockDim.x);
    const int smem = static_cast<int>(cfg.dynamicSmemBytes);
    const auto key = std::make_tuple(dev, fn, threads, smem, split <= 1 ? 1u : split);
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_occ.find(key);
        if (it != g_occ.end()) return static_cast<uint64_t>(it->second);
    }
    int n = 0;
    if (split <= 1) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, static_cast<size_t>(smem)) != cudaSuccess)
            n = 0;
    } else {
        cudaLaunchConfig_t c = cfg;
        c.gridDim = dim3(split * 64u);
        if (cudaOccupancyMaxActiveClusters(&n, fn, &c) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    std::lock_guard<std::mutex> lk(g_mu);
    g_occ[key] = n;
    return static_cast<uint64_t>(n);
}

uint64_t blocks_per_sm(int dev, const void* fn, int threads, int smem) {
    cudaLaunchConfig_t c{};
    c.blockDim = dim3(static_cast<unsigned>(threads));
    c.dynamicSmemBytes = static_cast<size_t>(smem);
    return resident(dev, fn, c, 1);
}

// Clusters of `split` blocks (or single blocks) that can be resident at once.
uint64_t resident_clusters(int dev, const void* fn, const cudaLaunchConfig_t& cfg, uint32_t split, int sms) {
    if (split <= 1) return resident(dev, fn, cfg, 1) * static_cast<uint64_t>(sms);
    return resident(dev, fn, cfg, split);
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
// m_max is the most input rows one call takes (0: any number).
int validate_args(const void* W, int wt, const float* x, const float* y, const Shape& s, uint32_t split,
                  uint32_t rows_per_cta, uint32_t m_max = kMaxRows) {
    if (!valid_wt(wt)) return fail(REM_EINVAL, "rem_matvec: unknown weight type %d", wt);
    if (s.m == 0 || (m_max && s.m > m_max))
        return m_max ? fail(REM_EINVAL, "rem_matvec: m (%u) must be in 1..=%u", s.m, m_max)
                     : fail(REM_EINVAL, "rem_matvec_many: m (%u) must be >= 1", s.m);
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

// The engine (and with it the arithmetic) of a weight shape: the tensor-core
// kernel for Q6_K, the lanes-over-rows kernel otherwise.  Q6_K's sub-block
// decode is what limits the lanes-over-rows kernel from m = 2 up (at 128256 x
// 4096 it takes 108, 271 and 512 us at m = 1, 4 and 8 against 127, 150 and
// 161 us on the tensor cores); for Q8_0 and Q5_0 the lanes-over-rows kernel
// is well ahead at m <= 2 and the tensor cores pull ahead only from m = 4
// (Q5_0 16384 x 4096: 21 against 29 us at m = 1, 50 against 36 at m = 8), so
// they keep the lanes-over-rows kernel.  Like the split, it depends on
// (wtype, rows, k) only.
int auto_engine(int wt, uint64_t rows, uint32_t k) {
    (void)rows;
    (void)k;
    return wt == kQ6_K ? REM_ENGINE_TC : REM_ENGINE_SIMT;
}

// Input rows one launch of an engine takes.
uint32_t engine_rows(int engine, int wt) {
    return engine == REM_ENGINE_TC ? static_cast<uint32_t>(tc_max_mp(wt)) : static_cast<uint32_t>(kMaxRows);
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

// The schedule of a call (rem_schedule with defaults filled in).
struct Sched {
    uint32_t split = 0, rows_per_cta = 0;
    int layout = -1, engine = -1;
    uint64_t wait_ns = 0;
    uint32_t test_flags = 0;
    uint32_t m_max = kMaxRows;  // input rows the entry point takes per launch
};

constexpr uint64_t kDefaultWaitNs = 10ull * 1000ull * 1000ull * 1000ull;  // 10 s per wait

// Schedule defaults of the calling thread (rem_set_thread_schedule).
thread_local bool g_thread_sched_set = false;
thread_local rem_schedule g_thread_sched;

// The schedule a call starts from: the thread's defaults where set.
Sched base_sched() {
    Sched sc;
    if (g_thread_sched_set) {
        sc.split = g_thread_sched.split;
        sc.rows_per_cta = g_thread_sched.rows_per_cta;
        sc.layout = g_thread_sched.layout;
        sc.engine = g_thread_sched.engine;
        sc.wait_ns = g_thread_sched.wait_ns;
        sc.test_flags = g_thread_sched.test_flags;
    }
    return sc;
}

// Schedule fields in range (host-only check).
int check_schedule(const rem_schedule& r) {
    if (r.layout < -1 || r.layout >= kNumLayouts)
        return fail(REM_EINVAL, "rem_matvec: layout (%d) must be -1 (auto) or 0..%d", r.layout, kNumLayouts - 1);
    if (r.engine < -1 || r.engine > REM_ENGINE_TC)
        return fail(REM_EINVAL, "rem_matvec: engine (%d) must be -1 (auto), %d or %d", r.engine, REM_ENGINE_SIMT,
                    REM_ENGINE_TC);
    if (r.split > REM_MAX_SPLIT)
        return fail(REM_EINVAL, "rem_matvec: split (%u) must be 0 (auto) or in 1..=%d", r.split, REM_MAX_SPLIT);
    if (!(r.rows_per_cta == 0 || r.rows_per_cta == 32 || r.rows_per_cta == 64 || r.rows_per_cta == 128))
        return fail(REM_EINVAL, "rem_matvec: rows_per_cta (%u) must be 0, 32, 64 or 128", r.rows_per_cta);
    return REM_OK;
}

// A launch plan: everything that follows from the shape, the schedule and
// the alignment of W, but not from the buffers' addresses (cached).
struct Plan {
    const void* fn = nullptr;
    int engine = REM_ENGINE_SIMT;
    int nr0 = 1, h = 1, warps = 4, stages = 2, smem = 0, threads = 0, mp = 8;
    uint32_t S = 1, cpb = 0, grid = 0, nchunk = 0;
    bool aligned = false, pdl = false, x_bm = false;
    bool cm = false;     // tensor-core engine: the MMA warps convert the inputs (tc_conv_mma)
    char note[96] = "";  // planner diagnostics (tensor-core engine: CTAs per SM for each ring depth)
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

using PlanKey = std::tuple<int, int, uint32_t, uint32_t, uint32_t, uint32_t, uint32_t, uint32_t, uint32_t,
                           uint32_t, uint32_t, uint32_t, int, int, bool>;
std::map<PlanKey, Plan> g_plans;

// When fewer CTAs run than can be resident, the block scheduler fills SMs to
// their occupancy limit and leaves others idle.  Asking for more (unused)
// shared memory per CTA caps the CTAs per SM at the even share, ceil(ctas /
// SMs), which spreads the grid over the SMs -- kept only if the whole grid
// still fits at once.
int spread_smem(int dev, const DeviceState& ds, const void* fn, cudaLaunchConfig_t cfg, uint32_t S, uint64_t ncl,
                int smem) {
    const uint64_t per_sm = (ncl * S + ds.sms - 1) / ds.sms;
    const uint64_t share = static_cast<uint64_t>(ds.smem_per_sm) / per_sm;
    if (share <= 1024u + static_cast<uint64_t>(smem)) return smem;
    const int cap = static_cast<int>(std::min<uint64_t>(static_cast<uint64_t>(ds.smem_optin), share - 1024u));
    if (cap <= smem || blocks_per_sm(dev, fn, static_cast<int>(cfg.blockDim.x), smem) <= per_sm) return smem;
    cfg.dynamicSmemBytes = static_cast<size_t>(cap);
    return resident_clusters(dev, fn, cfg, S, ds.sms) >= ncl ? cap : smem;
}

// Plan of the lanes-over-rows kernel: lane layout (NR0 rows per lane and H
// lane groups), row-block width G (consumer warps per CTA) and ring depth D:
// the fitting combination with the best score.  The score models a kernel
// that is bound by how many consumer warps each SM keeps busy (latency of
// shared-memory loads and stage waits): the average consumer warps per SM
// (saturating at 8), times the lane layout's weight (layout_weight), a single
// stage (no copy / compute overlap) 0.7x, the producer warp's share
// (G/(G+1))^2, 20% less per stage beyond two (deeper rings cost residency for
// no gain), all scaled by the share of resident CTA slots the last wave of
// row blocks keeps busy.  The weights were fitted to timings of every
// (layout, G, D) on GB300 for the five formats at 4096..128256 rows.
int plan_simt(int dev, const DeviceState& ds, int wt, const Shape& s, const Sched& sc, Plan& p) {
    const uint32_t S = p.S;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    if (S > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = S;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.numAttrs = 1;
    }
    double best = -1.0;
    int last_cap = 0;
    const int km = static_cast<int>(s.m);  // the kernel's M
    for (int l = kNumLayouts - 1; l >= 0; --l) {
        const void* f = mv_kernel(wt, km, l);
        if (!f || (sc.layout >= 0 && l != sc.layout)) continue;
        const int nr0 = layout_nr0(l), h = layout_h(l);
        const uint32_t rpw = static_cast<uint32_t>(kLanes * nr0);
        const int cap = ds.max_threads[wt][km][l];
        for (int g = kMaxWarps; g >= 1; g /= 2) {
            if (sc.rows_per_cta ? static_cast<uint32_t>(g) * rpw != sc.rows_per_cta
                                : (g > 4 || static_cast<uint32_t>(g) * rpw > 256u))
                continue;
            if ((g + 1) * 32 > cap) {
                last_cap = cap;
                continue;
            }
            const uint64_t nb = static_cast<uint64_t>(s.batch) * ((s.n + rpw * g - 1) / (rpw * g));
            const uint64_t units = nb * S;
            const uint64_t per_cta = ((p.nchunk + S - 1) / S) * ((units + 2ull * ds.sms - 1) / (2ull * ds.sms));
            const int dmax = static_cast<int>(std::min<uint64_t>(kMaxStages, std::max<uint64_t>(2, per_cta)));
            for (int d = 1; d <= dmax; ++d) {
                const int sm = static_cast<int>(mv_smem_bytes(wt, nr0, h, g, d, km, S));
                if (sm > ds.smem_optin) continue;
                cfg.blockDim = dim3(static_cast<unsigned>((g + 1) * 32));
                cfg.dynamicSmemBytes = static_cast<size_t>(sm);
                const uint64_t slots = resident_clusters(dev, f, cfg, S, ds.sms) * S;
                if (slots == 0) continue;
                const uint64_t ctas = std::min(units, slots);
                const uint64_t waves = (units + ctas - 1) / ctas;
                const double eff = static_cast<double>(units) / static_cast<double>(waves * ctas);
                const double warps_sm = static_cast<double>(ctas) / ds.sms * g;
                const double gf = static_cast<double>(g) / (g + 1);
                double score = std::min(warps_sm, 8.0) * layout_weight(wt, km, nr0, h) *
                               (d == 1 ? 0.7 : 1.0) * gf * gf * (1.0 - 0.2 * std::max(0, d - 2)) * eff;
                if (score > best) {
                    best = score;
                    p.fn = f;
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
        if (sc.layout >= 0 && !mv_kernel(wt, km, sc.layout))
            return fail(REM_ELAUNCH, "rem_matvec: lane layout %d has no %s kernel for m = %u", sc.layout,
                        wt_name(wt), s.m);
        if (last_cap)
            return fail(REM_ELAUNCH, "rem_matvec: %u rows per block exceed the %s kernel's limit of %d threads",
                        sc.rows_per_cta, wt_name(wt), last_cap);
        return fail(REM_ELAUNCH, "rem_matvec: no %s row block fits the device's shared memory", wt_name(wt));
    }
    const uint32_t rows_per_warp = static_cast<uint32_t>(kLanes * p.nr0);
    p.cpb = (s.n + rows_per_warp * p.warps - 1) / (rows_per_warp * p.warps);
    p.threads = (p.warps + 1) * 32;
    cfg.blockDim = dim3(static_cast<unsigned>(p.threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(p.smem);
    const uint64_t nblocks = static_cast<uint64_t>(p.cpb) * s.batch;
    const uint64_t res = resident_clusters(dev, p.fn, cfg, S, ds.sms);
    if (res == 0)
        return fail(REM_ELAUNCH, "rem_matvec: a cluster of %u blocks of %d threads and %d bytes does not fit", S,
                    p.threads, p.smem);
    const uint64_t ncl = std::min<uint64_t>(nblocks, res);
    if (ncl < res) p.smem = spread_smem(dev, ds, p.fn, cfg, S, ncl, p.smem);
    p.grid = static_cast<uint32_t>(ncl * S);
    return REM_OK;
}

// Plan of the tensor-core kernel: 128-row tiles, MP input rows per launch,
// the deepest stage ring (2..4) that keeps the most CTAs resident, and at
// most 512 / (tensor-memory columns) CTAs per SM: the tensor memory a CTA
// allocates must always be free when it starts, so the shared memory request
// is raised until no more CTAs than that fit on one SM.
int plan_tc(int dev, const DeviceState& ds, int wt, const Shape& s, Plan& p) {
    const uint32_t S = p.S;
    p.mp = tc_tile_mp(s.m);
    p.cm = tc_conv_mma(wt, s.m);
    p.fn = tc_kernel(wt, p.mp, p.cm);
    if (!p.fn || p.mp > tc_max_mp(wt))
        return fail(REM_ELAUNCH, "rem_matvec: no %s tensor-core kernel for m = %u", wt_name(wt), s.m);
    p.threads = tc_threads(p.mp);
    p.warps = tc_consumer_warps(p.mp);
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    if (S > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = S;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.numAttrs = 1;
    }
    cfg.blockDim = dim3(static_cast<unsigned>(p.threads));
    const uint64_t tmem_cap = 512u / static_cast<uint32_t>(tc_tmem_cols(wt, p.mp));
    uint64_t best_sm = 0;
    p.stages = 0;
    p.note[0] = '\0';
    for (int d = kMaxStages; d >= 2; --d) {
        const int sm = static_cast<int>(tc_smem_bytes(wt, p.mp, d, static_cast<int>(S)));
        if (sm > ds.smem_optin) continue;
        const uint64_t occ = blocks_per_sm(dev, p.fn, p.threads, sm);
        const size_t used = strlen(p.note);
        snprintf(p.note + used, sizeof(p.note) - used, " d%d:%dB/%llu", d, sm, static_cast<unsigned long long>(occ));
        const uint64_t per_sm = std::min(occ, tmem_cap);
        if (per_sm > best_sm) {
            best_sm = per_sm;
            p.stages = d;
            p.smem = sm;
        }
    }
    if (p.stages == 0 || best_sm == 0)
        return fail(REM_ELAUNCH, "rem_matvec: no %s tensor-core stage ring fits the device's shared memory",
                    wt_name(wt));
    if (blocks_per_sm(dev, p.fn, p.threads, p.smem) > tmem_cap) {
        const int need = ds.smem_per_sm / static_cast<int>(tmem_cap + 1) + 1;
        if (need > ds.smem_optin || blocks_per_sm(dev, p.fn, p.threads, need) > tmem_cap)
            return fail(REM_ELAUNCH, "rem_matvec: cannot hold %s tensor-core CTAs to %llu per SM", wt_name(wt),
                        static_cast<unsigned long long>(tmem_cap));
        p.smem = std::max(p.smem, need);
    }
    p.cpb = (s.n + kTcRows - 1) / kTcRows;
    cfg.dynamicSmemBytes = static_cast<size_t>(p.smem);
    const uint64_t nblocks = static_cast<uint64_t>(p.cpb) * s.batch;
    const uint64_t res = resident_clusters(dev, p.fn, cfg, S, ds.sms);
    if (res == 0)
        return fail(REM_ELAUNCH, "rem_matvec: a cluster of %u tensor-core blocks of %d bytes does not fit", S, p.smem);
    const uint64_t ncl = std::min<uint64_t>(nblocks, res);
    if (ncl < res) p.smem = spread_smem(dev, ds, p.fn, cfg, S, ncl, p.smem);
    p.grid = static_cast<uint32_t>(ncl * S);
    return REM_OK;
}

// Tensor maps, cached by everything they encode (the buffers' addresses
// included); a cache that grows past its bound is cleared.
struct MapKey {
    const void* ptr;
    uint32_t kind;
    cuuint64_t d0, d1, d2, s0, s1;
    cuuint32_t b0, b1, b2;
    bool operator<(const MapKey& o) const {
        return std::tie(ptr, kind, d0, d1, d2, s0, s1, b0, b1, b2) <
               std::tie(o.ptr, o.kind, o.d0, o.d1, o.d2, o.s0, o.s1, o.b0, o.b1, o.b2);
    }
};
std::map<MapKey, CUtensorMap> g_maps;

bool encode_map(CUtensorMap* out, CUtensorMapDataType dt, uint32_t rank, void* ptr, const cuuint64_t* dims,
                const cuuint64_t* strides, const cuuint32_t* box) {
    MapKey key{ptr, static_cast<uint32_t>(dt) * 8u + rank, dims[0], rank > 1 ? dims[1] : 0, rank > 2 ? dims[2] : 0,
               rank > 1 ? strides[0] : 0, rank > 2 ? strides[1] : 0, box[0], rank > 1 ? box[1] : 0,
               rank > 2 ? box[2] : 0};
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_maps.find(key);
        if (it != g_maps.end()) {
            *out = it->second;
            return true;
        }
    }
    const cuuint32_t estride[3] = {1, 1, 1};
    if (driver().encode(out, dt, rank, ptr, dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_maps.size() >= 1024) g_maps.clear();
    g_maps[key] = *out;
    return true;
}

int launch_matvec(const void* W, int wt, const float* x, float* y, const Shape& s, const Sched& sc, void* stream,
                  const Epilogue& epi = Epilogue(), const AffineArgs* aff = nullptr) {
    const int engine = sc.engine >= 0 ? sc.engine : auto_engine(wt, static_cast<uint64_t>(s.batch) * s.n, s.k);
    if (engine != REM_ENGINE_SIMT && engine != REM_ENGINE_TC)
        return fail(REM_EINVAL, "rem_matvec: engine (%d) must be -1 (auto), %d or %d", engine, REM_ENGINE_SIMT,
                    REM_ENGINE_TC);
    if (engine == REM_ENGINE_TC && !tc_format(wt))
        return fail(REM_EINVAL, "rem_matvec: the tensor-core engine takes Q8_0, Q5_0 and Q6_K weights, not %s",
                    wt_name(wt));
    int rc = validate_args(W, wt, x, y, s, sc.split, sc.rows_per_cta, std::min(sc.m_max, engine_rows(engine, wt)));
    if (rc != REM_OK) return rc;
    if (is_affine(wt) && !aff)
        return fail(REM_EINVAL, "rem_matvec: %s weights need their scales and biases: use rem_matvec_affine",
                    wt_name(wt));
    if (!is_affine(wt) && aff) return fail(REM_EINVAL, "rem_matvec_affine: %s is not an affine type", wt_name(wt));
    const uint64_t rb = row_bytes_of(wt, s.k);
    const uint64_t rows = static_cast<uint64_t>(s.batch) * s.n;
    DeviceState* ds = nullptr;
    int dev = 0;
    if ((rc = device_state(&ds, &dev)) != REM_OK) return rc;
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
    const uint32_t S = sc.split ? sc.split : auto_split(wt, rows, s.k);
    if (S > static_cast<uint32_t>(kMaxSplit))
        return fail(REM_ELAUNCH,
                    "rem_matvec: split %u needs clusters of %u thread blocks but the %s kernels launch clusters of "
                    "at most %d",
                    S, S, wt_name(wt), kMaxSplit);
    // Inputs: [batch][m][k] f32 with the caller's strides, dimensions ordered
    // by increasing stride; either order stages the box as [m][chunk].
    const uint64_t xrs = s.m == 1 ? s.k : s.xrs;
    const uint64_t xbs = s.batch == 1 ? xrs * s.m : s.xbs;
    const bool w_tma = reinterpret_cast<uintptr_t>(W) % 16 == 0 && rb % 16 == 0 && rows < (1ull << 31) &&
                       rb / 2 < (1ull << 32) && driver().encode != nullptr && xrs > 0 && xbs > 0;

    const PlanKey key{dev, wt, s.m, s.n, s.k, s.batch, s.xrs, s.xbs, s.yrs, s.ybs, S, sc.rows_per_cta, sc.layout,
                      engine, w_tma};
    Plan p;
    bool cached = false;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_plans.find(key);
        if (it != g_plans.end()) {
            p = it->second;
            cached = true;
        }
    }
    if (!cached) {
        p.engine = engine;
        p.S = S;
        p.nchunk = (s.k + chunk_values(wt) - 1) / chunk_values(wt);
        p.aligned = w_tma;
        p.x_bm = xbs < xrs;
        rc = engine == REM_ENGINE_TC ? plan_tc(dev, *ds, wt, s, p) : plan_simt(dev, *ds, wt, s, sc, p);
        if (rc != REM_OK) return rc;
        if (static_cast<uint64_t>(p.cpb) * s.batch > 0x7FFFFFFFull)
            return fail(REM_EINVAL, "rem_matvec: too many row blocks");
        // Programmatic dependent launch: the kernel may start while the
        // previous kernel of the stream finishes (it waits for it,
        // griddepcontrol.wait, before reading x or W into shared memory and
        // before writing y), and prefetches its first weights into L2
        // meanwhile.  That pays where the launch is short next to its
        // start-up latency -- from m = 4 up (compute bound) below 256 MB of
        // weights, at any m below 24 MB -- and costs throughput on long
        // bandwidth-bound launches, which keep plain stream order.
        // Scheduling only: the arithmetic is the same either way.
        const uint64_t wbytes = rb * rows;
        p.pdl = engine == REM_ENGINE_TC ? wbytes <= (64ull << 20)
                                        : ((s.m >= 4 && wbytes <= (256ull << 20)) || wbytes <= (24ull << 20));
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_plans.size() >= 4096) g_plans.clear();
        g_plans[key] = p;
    }

    alignas(64) CUtensorMap wmap, xmap;
    std::memset(&wmap, 0, sizeof(wmap));
    std::memset(&xmap, 0, sizeof(xmap));
    bool aligned = p.aligned;
    if (aligned) {
        const cuuint64_t gdim[3] = {s.k, p.x_bm ? s.batch : s.m, p.x_bm ? s.m : s.batch};
        const cuuint64_t gstride[2] = {4 * (p.x_bm ? xbs : xrs), 4 * (p.x_bm ? xrs : xbs)};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(chunk_values(wt)), p.x_bm ? 1u : s.m,
                                   p.x_bm ? s.m : 1u};
        aligned = encode_map(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(x), gdim, gstride, box);
    }
    if (aligned) {
        // weights as [rows][row_bytes/2] u16, one box = the row block's rows x one chunk
        const uint32_t brows = p.engine == REM_ENGINE_TC ? static_cast<uint32_t>(kTcRows)
                                                         : static_cast<uint32_t>(kLanes * p.nr0 * p.warps);
        const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(rb / 2), static_cast<cuuint64_t>(rows)};
        const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(rb)};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(chunk_box(wt) / 2), brows};
        aligned = encode_map(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(W), gdim, gstride, box);
    }
    snprintf(g_plan, sizeof(g_plan),
             "%s engine=%s m=%u n=%u k=%u batch=%u split=%u nr0=%d h=%d warps=%d mp=%d%s stages=%d smem=%d grid=%u "
             "row_blocks=%llu tma=%d pdl=%d occ=[%s ]",
             wt_name(wt), p.engine == REM_ENGINE_TC ? "tc" : "simt", s.m, s.n, s.k, s.batch, p.S, p.nr0, p.h, p.warps,
             p.mp, p.engine == REM_ENGINE_TC ? (p.cm ? " xconv=mma" : " xconv=consumers") : "", p.stages, p.smem, p.grid, static_cast<unsigned long long>(p.cpb) * s.batch,
             static_cast<int>(aligned), static_cast<int>(p.pdl), p.note);

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
    a.split = p.S;
    a.nchunk = p.nchunk;
    a.cpb = p.cpb;
    a.batch = s.batch;
    a.stages = static_cast<uint32_t>(p.stages);
    a.aligned = aligned ? 1u : 0u;
    a.x_bm = p.x_bm ? 1u : 0u;
    a.pdl = p.pdl ? 1u : 0u;
    a.m = s.m;
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
    a.status = ds->status;
    a.wait_ns = sc.wait_ns ? sc.wait_ns : kDefaultWaitNs;
    a.test_flags = sc.test_flags;

    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[2];
    cfg.stream = static_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    if (p.S > 1) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
        attr[cfg.numAttrs].val.clusterDim.x = p.S;
        attr[cfg.numAttrs].val.clusterDim.y = 1;
        attr[cfg.numAttrs].val.clusterDim.z = 1;
        ++cfg.numAttrs;
    }
    if (p.pdl) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
        ++cfg.numAttrs;
    }
    cfg.blockDim = dim3(static_cast<unsigned>(p.threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(p.smem);
    cfg.gridDim = dim3(p.grid);
    void* args[3] = {&wmap, &xmap, &a};
    const cudaError_t e = cudaLaunchKernelExC(&cfg, p.fn, args);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(REM_ECUDA, "rem_matvec: launch failed: %s", cudaGetErrorString(e));
    }
    return REM_OK;
}

// Any number of input rows: launches of up to the engine's rows each, one
// pass over W per launch.  Every rule for the whole call (output aliasing
// over all m rows included) and every group's rules are checked before the
// first launch.
int launch_many(const void* W, int wt, const float* x, float* y, const Shape& all, const Sched& sc, void* stream,
                const AffineArgs* aff = nullptr) {
    int rc = validate_args(W, wt, x, y, all, sc.split, sc.rows_per_cta, 0);
    if (rc != REM_OK) return rc;
    const int engine = sc.engine >= 0 ? sc.engine : auto_engine(wt, static_cast<uint64_t>(all.batch) * all.n, all.k);
    const uint32_t per = engine_rows(engine, wt);
    for (uint32_t j0 = 0; j0 < all.m; j0 += per) {
        const Shape g{std::min<uint32_t>(per, all.m - j0), all.n, all.k, all.batch, all.xrs, all.xbs, all.yrs,
                      all.ybs};
        if ((rc = validate_args(W, wt, x + static_cast<uint64_t>(j0) * all.xrs,
                                y + static_cast<uint64_t>(j0) * all.yrs, g, sc.split, sc.rows_per_cta, per)) != REM_OK)
            return rc;
    }
    // the split comes from the shape, so every group (and an m = 1 call)
    // uses the same one
    Sched g_sc = sc;
    g_sc.split = sc.split ? sc.split : auto_split(wt, static_cast<uint64_t>(all.batch) * all.n, all.k);
    g_sc.engine = engine;
    g_sc.m_max = per;
    for (uint32_t j0 = 0; j0 < all.m; j0 += per) {
        const Shape g{std::min<uint32_t>(per, all.m - j0), all.n, all.k, all.batch, all.xrs, all.xbs, all.yrs,
                      all.ybs};
        rc = launch_matvec(W, wt, x + static_cast<uint64_t>(j0) * all.xrs, y + static_cast<uint64_t>(j0) * all.yrs, g,
                           g_sc, stream, Epilogue(), aff);
        if (rc != REM_OK) return rc;
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
    case kA3G32: return lo ? mv_kernel_a3g32_a(m, layout) : mv_kernel_a3g32_b(m, layout);
    case kA3G64: return lo ? mv_kernel_a3g64_a(m, layout) : mv_kernel_a3g64_b(m, layout);
    case kA3G128: return lo ? mv_kernel_a3g128_a(m, layout) : mv_kernel_a3g128_b(m, layout);
    case kA5G32: return lo ? mv_kernel_a5g32_a(m, layout) : mv_kernel_a5g32_b(m, layout);
    case kA5G64: return lo ? mv_kernel_a5g64_a(m, layout) : mv_kernel_a5g64_b(m, layout);
    case kA5G128: return lo ? mv_kernel_a5g128_a(m, layout) : mv_kernel_a5g128_b(m, layout);
    case kA6G32: return lo ? mv_kernel_a6g32_a(m, layout) : mv_kernel_a6g32_b(m, layout);
    case kA6G64: return lo ? mv_kernel_a6g64_a(m, layout) : mv_kernel_a6g64_b(m, layout);
    case kA6G128: return lo ? mv_kernel_a6g128_a(m, layout) : mv_kernel_a6g128_b(m, layout);
    default: return nullptr;
    }
}

const void* tc_kernel(int wt, int mp, bool cm) {
    switch (wt) {
    case kQ8_0: return tc_kernel_q8_0(mp, cm);
    case kQ5_0: return tc_kernel_q5_0(mp, cm);
    case kQ6_K: return tc_kernel_q6_k(mp, cm);
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
    return launch_matvec(W, wtype, x, y, s, base_sched(), stream);
}

int rem_matvec_ex(const void* W, int wtype, uint32_t n, uint32_t k, uint32_t batch, const float* x, uint32_t m,
                  uint32_t x_row_stride, uint32_t x_batch_stride, float* y, uint32_t y_row_stride,
                  uint32_t y_batch_stride, uint32_t split, uint32_t rows_per_cta, void* stream) {
    g_err[0] = '\0';
    const Shape s{m, n, k, batch, x_row_stride, x_batch_stride, y_row_stride, y_batch_stride};
    Sched sc = base_sched();
    if (split) sc.split = split;
    if (rows_per_cta) sc.rows_per_cta = rows_per_cta;
    return launch_matvec(W, wtype, x, y, s, sc, stream);
}

int rem_matvec_sched(const void* W, int wtype, uint32_t n, uint32_t k, uint32_t batch, const float* x, uint32_t m,
                     uint32_t x_row_stride, uint32_t x_batch_stride, float* y, uint32_t y_row_stride,
                     uint32_t y_batch_stride, const rem_schedule* sched, void* stream) {
    g_err[0] = '\0';
    const Shape s{m, n, k, batch, x_row_stride, x_batch_stride, y_row_stride, y_batch_stride};
    Sched sc = base_sched();
    if (sched) {
        int rc = check_schedule(*sched);
        if (rc != REM_OK) return rc;
        if (sched->split) sc.split = sched->split;
        if (sched->rows_per_cta) sc.rows_per_cta = sched->rows_per_cta;
        if (sched->layout >= 0) sc.layout = sched->layout;
        if (sched->engine >= 0) sc.engine = sched->engine;
        if (sched->wait_ns) sc.wait_ns = sched->wait_ns;
        sc.test_flags |= sched->test_flags;
    }
    return launch_many(W, wtype, x, y, s, sc, stream);
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
    return launch_matvec(W, wtype, x, y, s, base_sched(), stream, e);
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
    Sched sc = base_sched();
    if (split) sc.split = split;
    return launch_matvec(codes, wtype, x, y, s, sc, stream, Epilogue(), &aff);
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
    Sched sc = base_sched();
    if (split) sc.split = split;
    return launch_many(W, wtype, x, y, all, sc, stream);
}

int rem_set_thread_schedule(const rem_schedule* sched) {
    if (!sched) {
        g_thread_sched_set = false;
        return REM_OK;
    }
    int rc = check_schedule(*sched);
    if (rc != REM_OK) return rc;
    g_thread_sched = *sched;
    g_thread_sched_set = true;
    return REM_OK;
}

int rem_engine_of(int wtype, uint32_t rows, uint32_t k) {
    if (!valid_wt(wtype) || rows == 0 || k == 0) return -1;
    return auto_engine(wtype, rows, k);
}

int rem_device_status(int clear) {
    g_err[0] = '\0';
    DeviceState* ds = nullptr;
    int dev = 0;
    int rc = device_state(&ds, &dev);
    if (rc != REM_OK) return rc;
    uint32_t word = 0;
    if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof(word)) != cudaSuccess) {
        cudaGetLastError();
        return fail(REM_ECUDA, "rem_device_status: cannot read the status word of device %d", dev);
    }
    if (clear && word != 0) {
        const uint32_t zero = 0;
        if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess) {
            cudaGetLastError();
            return fail(REM_ECUDA, "rem_device_status: cannot clear the status word of device %d", dev);
        }
    }
    if (word & kStatusWaitTimeout)
        return fail(REM_ECUDA,
                    "rem_device_status: a kernel on device %d gave up on a bounded wait; the outputs it could not "
                    "finish hold NaN",
                    dev);
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

const char* rem_last_plan(void) { return g_plan; }

int rem_version(void) { return 2; }

}  // extern "C"
