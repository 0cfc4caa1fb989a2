// rem_internal.h -- declarations shared by the host library and the kernels.
//
// Weight formats follow mlx-native 0.18.0 src/ops/row_exact_matvec.rs
// (RowExactWeight: F16, Q8_0, Q4_K, Q6_K, Q5_0 and their block sizes).
#pragma once
#include <cstdint>

namespace rem {

enum Wt : int {
    kF16 = 0, kQ8_0 = 1, kQ4_K = 2, kQ6_K = 3, kQ5_0 = 4, kF32 = 5, kBF16 = 6,
    // affine group quantization: 3-, 4-, 5-, 6- or 8-bit codes, binary16 scale and bias per group of
    // 32/64/128 values
    kA4G32 = 7, kA4G64 = 8, kA4G128 = 9, kA8G32 = 10, kA8G64 = 11, kA8G128 = 12,
    kA3G32 = 13, kA3G64 = 14, kA3G128 = 15, kA5G32 = 16, kA5G64 = 17, kA5G128 = 18,
    kA6G32 = 19, kA6G64 = 20, kA6G128 = 21,
    kNumWt = 22
};
__host__ __device__ constexpr bool is_affine(int wt) {
    return (wt >= kA4G32 && wt <= kA8G128) || (wt >= kA3G32 && wt <= kA6G128);
}
__host__ __device__ constexpr int affine_bits(int wt) {
    return wt <= kA4G128 ? 4 : wt <= kA8G128 ? 8 : wt <= kA3G128 ? 3 : wt <= kA5G128 ? 5 : 6;
}
// the affine types come in triples of group sizes 32, 64, 128
__host__ __device__ constexpr int affine_group(int wt) {
    return 32 << ((wt - (wt >= kA3G32 ? kA3G32 : kA4G32)) % 3);
}

constexpr int kMaxRows = 8;        // ROW_EXACT_MATVEC_MAX_ROWS
constexpr int kLanes = 32;         // weight rows per warp and NR0: one row per lane
constexpr int kMaxWarps = 4;       // consumer warps per CTA (kernels are bounded to 5 warps)
constexpr int kMaxSplit = 8;       // K ranges per row = CTAs per cluster (portable cluster limit)
constexpr int kMaxStages = 4;      // pipeline stages (mbarriers) per warp

// Values and bytes of one block (the *_BLOCK_VALUES / *_BLOCK_BYTES constants).
// (An affine "block" is one group's codes; its scale and bias live in their own arrays.)
__host__ __device__ constexpr int block_values(int wt) {
    return is_affine(wt) ? affine_group(wt)
           : (wt == kF16 || wt == kF32 || wt == kBF16) ? 1 : (wt == kQ8_0 || wt == kQ5_0) ? 32 : 256;
}
__host__ __device__ constexpr int block_bytes(int wt) {
    return is_affine(wt) ? affine_group(wt) * affine_bits(wt) / 8
           : (wt == kF16 || wt == kBF16) ? 2 : wt == kF32 ? 4 : wt == kQ8_0 ? 34 : wt == kQ5_0 ? 22
           : wt == kQ4_K ? 144 : 210;
}

// Staging geometry.  A "chunk" is the slice of one weight row a lane decodes
// between two pipeline waits: 72 F16 or BF16 values, 36 F32 values, 4 Q8_0
// blocks, 8 Q5_0 blocks, one Q4_K / Q6_K super-block, 128 bytes of 4- or
// 8-bit affine codes (256 / 128 values, staged as a 144-byte window), or 256
// 3-, 5- or 6-bit affine codes (96, 160 or 192 bytes, staged as 112-, 176-
// or 208-byte windows).  A warp stages the same chunk of its 32*NR0
// rows as one 2-D TMA box, one row every `box` bytes.  Box widths are odd
// multiples of 16 bytes, so 32 lanes reading 16 bytes each at the same
// offset of their own rows hit distinct bank quads (4 wavefronts, the
// minimum).  Q8_0 and Q6_K stage the 16-byte aligned window (144 / 240
// bytes) around their 136 / 210 chunk bytes.
__host__ __device__ constexpr int chunk_values(int wt) {
    return is_affine(wt) ? ((affine_bits(wt) == 4 || affine_bits(wt) == 8) ? 1024 / affine_bits(wt) : 256)
           : (wt == kF16 || wt == kBF16) ? 72 : wt == kF32 ? 36 : wt == kQ8_0 ? 128 : 256;
}
__host__ __device__ constexpr int chunk_box(int wt) {
    return is_affine(wt) ? (affine_bits(wt) == 3 ? 112 : affine_bits(wt) == 5 ? 176 : affine_bits(wt) == 6 ? 208 : 144)
           : (wt == kF16 || wt == kBF16 || wt == kF32 || wt == kQ8_0 || wt == kQ4_K) ? 144
           : wt == kQ5_0 ? 176 : 240;
}

// Kernel argument block (one launch).  Grid: a number of clusters of
// `split` CTAs that walk the batch * cpb row blocks; CTA rank s of a cluster
// handles K range s.
struct MvArgs {
    const uint8_t* w;        // weight rows, batch b at b*n*row_bytes
    const float* x;          // input, element (b, j, k) at b*xbs + j*xrs + k
    float* y;                // output, element (b, j, i) at b*ybs + j*yrs + i
    uint64_t row_bytes;
    uint32_t n, k;
    uint32_t xrs, xbs, yrs, ybs;
    uint32_t split;          // K ranges per row = CTAs per cluster (fixes the reduction order)
    uint32_t nchunk;         // chunks per row
    uint32_t cpb;            // row blocks per batch (each covers warps*32*NR0 rows)
    uint32_t batch;
    uint32_t stages;         // pipeline stages (1..4)
    uint32_t aligned;        // 1: TMA staging (16-byte aligned rows, encodable input map)
    uint32_t x_bm;           // input map dimension order: 1 = [k, batch, m] (token-major), 0 = [k, m, batch]
    uint32_t pdl;            // 1: launched as a programmatic dependent of the stream's previous kernel
    uint32_t m;              // input rows of the launch (the tensor-core kernel pads them to its MP)
    // epilogue: 0 = y = acc; 1 = y = alpha*acc; 2 = y = fma(alpha, acc, beta*c)
    uint32_t epi;
    float alpha, beta;
    const float* c;          // addend, element (b, j, i) at b*cbs + j*crs + i (read only when epi == 2)
    uint32_t crs, cbs;
    // affine weights: binary16 scale and bias of group g of global row r at r*ngroups + g
    const uint16_t* scales;
    const uint16_t* biases;
    uint32_t ngroups;
    // failure reporting: a wait that runs out after wait_ns nanoseconds ORs
    // kStatusWaitTimeout into *status and the launch writes NaN for the
    // outputs it could not finish
    uint32_t* status;
    uint64_t wait_ns;
    uint32_t test_flags;     // kTest* bits (test hooks; 0 in normal use)
};

// Bits of the device status word.
constexpr uint32_t kStatusWaitTimeout = 1u;  // a bounded wait ran out
// Test hooks (MvArgs::test_flags).
constexpr uint32_t kTestSkipFirstStage = 1u;  // no copy for the first pipeline stage (TMA staging)

// Lane layouts of the mat-vec kernel.  A warp always owns 32*nr0 weight
// rows; its lanes form h groups of 32/h lanes, each lane holding nr0*h of the
// warp's rows (lane l: rows l%(32/h) + (32/h)*i) and ceil(m/h) of the m
// input rows (group g: rows min(g*ceil(m/h), m - ceil(m/h)) onwards).  Every
// input value a lane loads from shared memory then feeds nr0*h weight rows.
constexpr int kNumLayouts = 4;
constexpr int layout_nr0(int l) { return (l == 1 || l == 3) ? 2 : 1; }
constexpr int layout_h(int l) { return l >= 2 ? 2 : 1; }

// Kernel lookup: rem_mv_kernel<wt, m, nr0, h> of layout index `layout`
// (0: nr0 1, h 1; 1: nr0 2, h 1; 2: nr0 1, h 2; 3: nr0 2, h 2), m in 1..8;
// nullptr where that kernel does not exist.
const void* mv_kernel(int wt, int m, int layout);
#define REM_DECLARE_PARTS(NAME) \
    const void* NAME##_a(int m, int layout); \
    const void* NAME##_b(int m, int layout);
REM_DECLARE_PARTS(mv_kernel_f16)
REM_DECLARE_PARTS(mv_kernel_q8_0)
REM_DECLARE_PARTS(mv_kernel_q5_0)
REM_DECLARE_PARTS(mv_kernel_q4_k)
REM_DECLARE_PARTS(mv_kernel_q6_k)
REM_DECLARE_PARTS(mv_kernel_f32)
REM_DECLARE_PARTS(mv_kernel_bf16)
REM_DECLARE_PARTS(mv_kernel_a4g32)
REM_DECLARE_PARTS(mv_kernel_a4g64)
REM_DECLARE_PARTS(mv_kernel_a4g128)
REM_DECLARE_PARTS(mv_kernel_a8g32)
REM_DECLARE_PARTS(mv_kernel_a8g64)
REM_DECLARE_PARTS(mv_kernel_a8g128)
REM_DECLARE_PARTS(mv_kernel_a3g32)
REM_DECLARE_PARTS(mv_kernel_a3g64)
REM_DECLARE_PARTS(mv_kernel_a3g128)
REM_DECLARE_PARTS(mv_kernel_a5g32)
REM_DECLARE_PARTS(mv_kernel_a5g64)
REM_DECLARE_PARTS(mv_kernel_a5g128)
REM_DECLARE_PARTS(mv_kernel_a6g32)
REM_DECLARE_PARTS(mv_kernel_a6g64)
REM_DECLARE_PARTS(mv_kernel_a6g128)
#undef REM_DECLARE_PARTS

// Dynamic shared memory of one CTA; the kernel lays it out the same way:
// stages x [weight box (warps*32*NR0 rows x box) | input box (m x chunk
// floats, padded to 128 B)], then the full and empty mbarriers of the
// stages, plus slack to align the base to 128 bytes.  With split > 1 two buffers of cross-range partial sums
// (one per row-block parity) sit between the stages and the mbarriers.
// `warps` counts consumer warps; the producer warp adds one more.
inline uint32_t mv_stage_bytes(int wt, int nr0, int warps, int m) {
    const uint32_t xb = (uint32_t)m * chunk_values(wt) * 4u;
    return (uint32_t)warps * kLanes * nr0 * chunk_box(wt) + ((xb + 127u) & ~127u);
}
inline uint32_t mv_smem_bytes(int wt, int nr0, int h, int warps, int stages, int m, int split) {
    const uint32_t mh = (uint32_t)((m + h - 1) / h);
    const uint32_t parts = split > 1 ? 2u * (uint32_t)warps * nr0 * h * mh * kLanes * 4u : 0u;
    return (uint32_t)stages * mv_stage_bytes(wt, nr0, warps, m) + parts + 16u * kMaxStages + 128u;
}

// ---------------------------------------------------------------- tensor-core engine

// The tensor-core kernel rem_tc_kernel<wt, mp, cm> (rem_tc.cuh) serves the
// block-scaled formats Q8_0, Q5_0 and Q6_K for up to mp input rows per
// launch, mp in {1, 2, 4, 8, 16, 32} (Q6_K: up to 16): a launch takes the
// smallest mp >= m, so the scaling of the accumulators handles exactly mp
// columns with no branch on m.  A CTA owns 128 weight rows.
// (Q4_K's weights d*sc*q - dmin*mn have no exact bfloat16 code, and the
// split a*sum(q*x) - b*sum(x) misses the tolerance where the two terms
// cancel and turns an infinite input into NaN, so Q4_K stays on the
// lanes-over-rows kernel, which dequantizes each weight exactly.)
constexpr int kTcRows = 128;
__host__ __device__ constexpr bool tc_format(int wt) { return wt == kQ8_0 || wt == kQ5_0 || wt == kQ6_K; }
// Q6_K's 16-value sub-blocks take twice the accumulator columns per unit, so
// its widest tile is 16 input rows; the formats with 32-value scale blocks go
// to 32.
__host__ __device__ constexpr int tc_max_mp(int wt) { return wt == kQ6_K ? 16 : 32; }
// MMA N: 2*mp columns (x_hi rows, x_lo rows), at least 16 (the rest of a
// narrow tile's B rows stay zero).
__host__ __device__ constexpr int tc_ncol(int mp) { return mp < 8 ? 16 : 2 * mp; }
// The tile width a launch of m input rows takes.
__host__ __device__ constexpr int tc_tile_mp(uint32_t m) {
    return m <= 1 ? 1 : m <= 2 ? 2 : m <= 4 ? 4 : m <= 8 ? 8 : m <= 16 ? 16 : 32;
}
// K-steps (16 values) per scale block: Q6_K sub-blocks of 16, Q8_0 / Q5_0 blocks of 32.
__host__ __device__ constexpr int tc_kpb(int wt) { return wt == kQ6_K ? 1 : 2; }
// K-steps of a 64-value unit each consumer warp decodes: two (8 consumer
// warps, two per lane quarter of the tile).  Every tile width takes the same
// warp assignment, so the arithmetic of an output does not depend on it.
__host__ __device__ constexpr int tc_kpw(int) { return 2; }
__host__ __device__ constexpr int tc_consumer_warps(int mp) { return 4 * (4 / tc_kpw(mp)); }
// consumers, the producer and two MMA warps
__host__ __device__ constexpr int tc_threads(int mp) { return (tc_consumer_warps(mp) + 3) * 32; }
// K-steps one accumulator region covers (the MMAs of a scale block's
// K-steps accumulate when one warp reads them all) and regions per unit.
__host__ __device__ constexpr int tc_region_ksteps(int wt, int mp) {
    return tc_kpw(mp) < tc_kpb(wt) ? tc_kpw(mp) : tc_kpb(wt);
}
__host__ __device__ constexpr int tc_regions(int wt, int mp) { return 4 / tc_region_ksteps(wt, mp); }
// Units of 64 values per staged chunk: Q8_0 2 (a chunk is 4 blocks), Q5_0 and Q6_K 4.
__host__ __device__ constexpr int tc_units_per_chunk(int wt) { return wt == kQ8_0 ? 2 : 4; }
// Whether the two MMA warps convert a chunk's inputs into its B tile (each
// the K-steps of its own units; 4 * units-per-chunk 16-byte items per input
// row between them) or the consumer warps do: the MMA warps while the items
// stay few enough for them, measured per format.  The conversion is the same
// arithmetic either way.
__host__ __device__ constexpr bool tc_conv_mma(int wt, uint32_t m) {
    return m * 4u * static_cast<uint32_t>(tc_units_per_chunk(wt)) <= (wt == kQ6_K ? 64u : 128u);
}
// Tensor-memory columns of one A/D slot: 32 columns of A (a unit as bf16
// pairs) and one N-column accumulator per region of the unit.
__host__ __device__ constexpr int tc_slot_cols(int wt, int mp) { return 32 + tc_regions(wt, mp) * tc_ncol(mp); }
// A/D slots in tensor memory: the deepest ring (4, 2 or 1 slots) that divides
// the units of a chunk and fits the SM's 512 columns (a tensor-core CTA runs
// alone on its SM).
__host__ __device__ constexpr int tc_slots(int wt, int mp) {
    return (tc_units_per_chunk(wt) % 4 == 0 && 4 * tc_slot_cols(wt, mp) <= 512) ? 4
           : (2 * tc_slot_cols(wt, mp) <= 512) ? 2 : 1;
}
// Tensor-memory columns a CTA allocates: its slots, rounded up to a power of two.
__host__ __device__ constexpr int tc_tmem_cols(int wt, int mp) {
    return (tc_slots(wt, mp) * tc_slot_cols(wt, mp)) <= 32    ? 32
           : (tc_slots(wt, mp) * tc_slot_cols(wt, mp)) <= 64  ? 64
           : (tc_slots(wt, mp) * tc_slot_cols(wt, mp)) <= 128 ? 128
           : (tc_slots(wt, mp) * tc_slot_cols(wt, mp)) <= 256 ? 256
                                                               : 512;
}
// Dynamic shared memory of one tensor-core CTA: stages x [weight box (128 rows
// x box) | input box (mp x chunk floats, padded to 128 B)], two B tiles of a
// chunk (bf16, N rows x chunk values), two buffers of partials (the warp
// groups past the first of each lane quarter, x 4 quarters x mp x 32 floats;
// the cross-range partials reuse them), the mbarriers and the tensor-memory
// address, plus slack to align the base to 128 bytes.
inline uint32_t tc_smem_bytes(int wt, int mp, int stages, int split) {
    const uint32_t xpad = ((uint32_t)mp * chunk_values(wt) * 4u + 127u) & ~127u;
    const uint32_t stage = (uint32_t)kTcRows * chunk_box(wt) + xpad;
    const uint32_t btiles = 2u * (uint32_t)(chunk_values(wt) / 16) * 32u * (uint32_t)tc_ncol(mp);
    const uint32_t groups = (uint32_t)tc_consumer_warps(mp) / 4u;
    const uint32_t pbuf = 2u * (groups - 1u) * 4u * (uint32_t)mp * 32u * 4u;
    (void)split;
    // mbarriers: full and empty per stage, A full and D full per step slot (4 + 4), a drain per
    // MMA warp, a B-buffer release per MMA warp and buffer (2 x 2)
    return (uint32_t)stages * stage + btiles + pbuf + 8u * (2 * kMaxStages + 4 + 4 + 2 + 4) + 16u + 128u;
}
const void* tc_kernel(int wt, int mp, bool cm);
const void* tc_kernel_q8_0(int mp, bool cm);
const void* tc_kernel_q5_0(int mp, bool cm);
const void* tc_kernel_q6_k(int mp, bool cm);

// Auxiliary kernels (dequantize / quantize), rem_aux.cu.
int launch_dequantize(const uint8_t* w, int wt, uint64_t rows, uint32_t k, uint64_t row_bytes,
                      float* out, void* stream);
int launch_dequantize_affine(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases, int wt,
                             uint64_t rows, uint32_t k, float* out, void* stream);
int launch_quantize(const float* src, int wt, uint64_t rows, uint32_t k, uint64_t row_bytes,
                    uint8_t* w, void* stream);

}  // namespace rem
