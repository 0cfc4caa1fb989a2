// rem_mv.cuh -- the row-exact few-row mat-vec kernel for sm_103a.
//
// y[b, j, i] = sum_k W[b*n + i, k] * x[b, j, k],  j < M <= 8
// (mlx-native 0.18.0 src/ops/row_exact_matvec.rs, module doc).
//
// Work mapping.  A warp owns 32*NR0 consecutive weight rows, one row per lane
// (lane l holds rows l and l+32).  All lanes of a warp work on the same K
// positions at the same time, so every input load is a shared-memory
// broadcast and every weight row is read from HBM exactly once for all M
// input rows.  K is cut into `split` contiguous ranges of chunks.  The
// `split` CTAs of a thread-block cluster share the same rows and take one
// range each; their partial sums are added in range order through
// distributed shared memory by the cluster's rank-0 CTA.  Each CTA streams
// its chunks through a ring of TMA stages: one box of weight rows and one box
// of the matching inputs per stage, completed on one mbarrier.
//
// Row exactness (module doc "Row exactness").  The arithmetic of output
// (i, j) depends only on row i's bytes, input row j and `split`:
//   * each block / sub-block u contributes through one packed chain
//     c = fma2(w[2p..2p+1], x[2p..2p+1], c) over its value pairs in order,
//   * then acc = fma2((a_u, a_u), c, acc) with the block scale a_u
//     (Q4_K also acc.x = fma(-min_u, sum(x of u), acc.x); F16 acc = acc + c),
//   * a range's partial is acc.x + acc.y, and ranges are summed in order.
// Nothing in that sequence depends on M, NR0, the CTA packing or the
// staging path, so row j of an M-row launch equals the same row of an M=1
// launch bit for bit.  fma.rn.f32x2 performs two independent, correctly
// rounded FMAs, identical to two scalar fmaf.
//
// Block decode.  Integer codes become exact floats without a conversion
// instruction: a code q placed in mantissa bits [p, p+w) under the exponent
// 2^(23-p) reads as 2^(23-p) + q, and one add of -(2^(23-p) + offset)
// yields q - offset exactly (offset 128 for int8 stored as uint8, 16 for
// Q5_0, 32 for Q6_K).
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cstdint>
#include <type_traits>

#include "rem_internal.h"

namespace rem {
namespace dev {

// ---------------------------------------------------------------- helpers

// Compile-time loop: f(std::integral_constant<int, I>) for I in [I0, N).
template <int I0, int N, typename F>
__device__ __forceinline__ void static_for(F&& f) {
    if constexpr (I0 < N) {
        f(std::integral_constant<int, I0>{});
        static_for<I0 + 1, N>(f);
    }
}

__device__ __forceinline__ float fbits(uint32_t u) { return __uint_as_float(u); }

__device__ __forceinline__ float h2f(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
}

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rc, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rc;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 ra, ra, rb;\n\t"
        "mov.b64 {%0, %1}, ra;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float4 ldg4(const float* p) {
    return __ldg(reinterpret_cast<const float4*>(p));
}

// Input values staged in shared memory (all lanes read the same address: a
// broadcast).
__device__ __forceinline__ float4 ldx4(const float* p) { return *reinterpret_cast<const float4*>(p); }

__device__ __forceinline__ uint4 lds16(const uint8_t* p) {
    return *reinterpret_cast<const uint4*>(p);
}

__device__ __forceinline__ uint32_t comp(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier / TMA

// Bounded wait: a phase that does not complete within the limit reports
// failure instead of spinning forever.
constexpr uint32_t kWaitLimit = 1u << 20;

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (uint32_t it = 0; it < kWaitLimit; ++it) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// ---------------------------------------------------------------- format traits

// Staged bytes per row (the TMA box width) and the byte position inside the
// staged row where chunk `cc` starts.
template <int WT> struct Stage;
template <> struct Stage<kF16> {
    static constexpr int kValues = 136, kBox = 272;
    __device__ static uint32_t gofs(uint32_t cc) { return cc * 272u; }  // global byte offset of the box
    __device__ static int sofs(uint32_t) { return 0; }
};
template <> struct Stage<kQ8_0> {
    static constexpr int kValues = 256, kBox = 272;
    __device__ static uint32_t gofs(uint32_t cc) { return cc * 272u; }
    __device__ static int sofs(uint32_t) { return 0; }
};
template <> struct Stage<kQ5_0> {
    static constexpr int kValues = 256, kBox = 176;
    __device__ static uint32_t gofs(uint32_t cc) { return cc * 176u; }
    __device__ static int sofs(uint32_t) { return 0; }
};
template <> struct Stage<kQ4_K> {
    static constexpr int kValues = 256, kBox = 144;
    __device__ static uint32_t gofs(uint32_t cc) { return cc * 144u; }
    __device__ static int sofs(uint32_t) { return 0; }
};
// Q6_K super-blocks (210 B) are only 2-byte aligned: stage the 16-byte
// aligned 240-byte window that contains super-block cc; it starts
// (210*cc) mod 16 bytes into the window (rows are 16-byte aligned whenever
// the TMA path is used, and the fallback copies to the same position).
template <> struct Stage<kQ6_K> {
    static constexpr int kValues = 256, kBox = 240;
    __device__ static uint32_t gofs(uint32_t cc) { return (cc * 210u) & ~15u; }
    __device__ static int sofs(uint32_t cc) { return static_cast<int>((cc * 210u) & 15u); }
};

// ---------------------------------------------------------------- decoders

// Q8_0 block B of a staged chunk (34 B at byte 34*B of a 16-aligned row).
// Yields the scale and the 16 code pairs as exact floats.
template <int B>
__device__ __forceinline__ void dec_q8_0(const uint8_t* row, float& d, float2 (&w)[16]) {
    constexpr int off = 34 * B, p0 = off >> 4, bo = off & 15;
    const uint4 v0 = lds16(row + 16 * p0), v1 = lds16(row + 16 * (p0 + 1)), v2 = lds16(row + 16 * (p0 + 2));
    const uint32_t W[12] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w, v2.x, v2.y, v2.z, v2.w};
    const uint32_t dw = W[bo >> 2];
    d = h2f((bo & 2) ? (dw >> 16) : dw);
#pragma unroll
    for (int p = 0; p < 16; ++p) {
        const int pos = bo + 2 + 2 * p;
        uint32_t v = W[pos >> 2];
        if (pos & 2) v >>= 16;
        // bytes biased by 128 (q + 128 in 0..255) under exponents 2^23, 2^15
        const float f0 = fbits(((v ^ 0x80u) & 0xFFu) | 0x4B000000u);
        const float f1 = fbits(((v ^ 0x8000u) & 0xFF00u) | 0x47000000u);
        w[p] = add2(make_float2(f0, f1), make_float2(-8388736.0f, -32896.0f));
    }
}

// 32-bit little-endian word at an even byte position of a word array.
template <int POS, int N>
__device__ __forceinline__ uint32_t u32_at(const uint32_t (&W)[N]) {
    if constexpr ((POS & 3) == 0) {
        return W[POS >> 2];
    } else {
        return __byte_perm(W[POS >> 2], W[(POS >> 2) + 1], 0x5432);
    }
}

// Spread the 4 low bits of h to bit 4 of each byte (bit k -> bit 8k+4).
__device__ __forceinline__ uint32_t spread4(uint32_t h) { return (h * 0x02040810u) & 0x10101010u; }

// Q5_0 block B (22 B at byte 22*B of a 16-aligned row).
template <int B>
__device__ __forceinline__ void dec_q5_0(const uint8_t* row, float& d, float2 (&w)[16]) {
    constexpr int off = 22 * B, p0 = off >> 4, bo = off & 15;
    const uint4 v0 = lds16(row + 16 * p0), v1 = lds16(row + 16 * (p0 + 1));
    uint4 v2 = make_uint4(0u, 0u, 0u, 0u);
    if constexpr (bo + 22 > 32) v2 = lds16(row + 16 * (p0 + 2));
    const uint32_t W[12] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w, v2.x, v2.y, v2.z, v2.w};
    const uint32_t dw = W[bo >> 2];
    d = h2f((bo & 2) ? (dw >> 16) : dw);
    const uint32_t qh = u32_at<bo + 2>(W);
    const uint32_t qs[4] = {u32_at<bo + 6>(W), u32_at<bo + 10>(W), u32_at<bo + 14>(W), u32_at<bo + 18>(W)};
    const float2 bias = make_float2(-8388624.0f, -32784.0f);  // 2^23 + 16, 2^15 + 16
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        // elements 4g..4g+3: low nibbles; elements 16+4g..: high nibbles
        const uint32_t lo = (qs[g] & 0x0F0F0F0Fu) | spread4((qh >> (4 * g)) & 0xFu);
        const uint32_t hi = ((qs[g] >> 4) & 0x0F0F0F0Fu) | spread4((qh >> (16 + 4 * g)) & 0xFu);
        const uint32_t lo2 = lo >> 16, hi2 = hi >> 16;
        w[2 * g] = add2(make_float2(fbits((lo & 0xFFu) | 0x4B000000u), fbits((lo & 0xFF00u) | 0x47000000u)), bias);
        w[2 * g + 1] = add2(make_float2(fbits((lo2 & 0xFFu) | 0x4B000000u), fbits((lo2 & 0xFF00u) | 0x47000000u)), bias);
        w[8 + 2 * g] = add2(make_float2(fbits((hi & 0xFFu) | 0x4B000000u), fbits((hi & 0xFF00u) | 0x47000000u)), bias);
        w[9 + 2 * g] = add2(make_float2(fbits((hi2 & 0xFFu) | 0x4B000000u), fbits((hi2 & 0xFF00u) | 0x47000000u)), bias);
    }
}

// Q4_K: 16 value pairs of sub-block 2c+H from the 8 qs words of chunk c.
// Low nibbles (H = 0) sit at bits 0, 8, 16 and (after >> 12) 12;
// high nibbles (H = 1) at bits 4, 12 and (after >> 12) 8, 16.
template <int H>
__device__ __forceinline__ void dec_q4_k_sub(const uint32_t (&q)[8], float2 (&w)[16]) {
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        const uint32_t v = q[g], s = v >> 12;
        if constexpr (H == 0) {
            w[2 * g] = add2(make_float2(fbits((v & 0xFu) | 0x4B000000u), fbits((v & 0xF00u) | 0x47000000u)),
                            make_float2(-8388608.0f, -32768.0f));
            w[2 * g + 1] = add2(make_float2(fbits((v & 0xF0000u) | 0x43000000u), fbits((s & 0xF000u) | 0x45000000u)),
                                make_float2(-128.0f, -2048.0f));
        } else {
            w[2 * g] = add2(make_float2(fbits((v & 0xF0u) | 0x49000000u), fbits((v & 0xF000u) | 0x45000000u)),
                            make_float2(-524288.0f, -2048.0f));
            w[2 * g + 1] = add2(make_float2(fbits((s & 0xF00u) | 0x47000000u), fbits((s & 0xF0000u) | 0x43000000u)),
                                make_float2(-32768.0f, -128.0f));
        }
    }
}

// 6-bit scale / min of Q4_K sub-block s from the 12 scale bytes (words s0, s1, s2).
__device__ __forceinline__ void q4k_scale_min(uint32_t s0, uint32_t s1, uint32_t s2, int s, uint32_t& sc,
                                              uint32_t& mn) {
    if (s < 4) {
        sc = (s0 >> (8 * s)) & 63u;
        mn = (s1 >> (8 * s)) & 63u;
    } else {
        const uint32_t b8 = (s2 >> (8 * (s - 4))) & 0xFFu;
        sc = (b8 & 0xFu) | (((s0 >> (8 * (s - 4) + 6)) & 3u) << 4);
        mn = (b8 >> 4) | (((s1 >> (8 * (s - 4) + 6)) & 3u) << 4);
    }
}

// Q6_K: the 53 little-endian words of a super-block (bytes 4i..4i+3, the
// last one holding only d) of a row staged with the super-block at byte O
// (even, < 16).  Only this load is specialised on O; the decode is shared.
template <int O>
__device__ __forceinline__ void q6_load_at(const uint8_t* row, uint32_t (&wd)[53]) {
    constexpr int wo = O >> 2;
    uint32_t P[60];
#pragma unroll
    for (int p = 0; p < 15; ++p) {
        const uint4 v = lds16(row + 16 * p);
        P[4 * p] = v.x; P[4 * p + 1] = v.y; P[4 * p + 2] = v.z; P[4 * p + 3] = v.w;
    }
#pragma unroll
    for (int i = 0; i < 53; ++i) {
        if constexpr ((O & 2) == 0) {
            wd[i] = P[wo + i];
        } else {
            wd[i] = __byte_perm(P[wo + i], P[wo + i + 1], 0x5432);
        }
    }
}

__device__ __forceinline__ void q6_load(const uint8_t* row, int o, uint32_t (&wd)[53]) {
    switch (o) {
    case 0: q6_load_at<0>(row, wd); break;
    case 2: q6_load_at<2>(row, wd); break;
    case 4: q6_load_at<4>(row, wd); break;
    case 6: q6_load_at<6>(row, wd); break;
    case 8: q6_load_at<8>(row, wd); break;
    case 10: q6_load_at<10>(row, wd); break;
    case 12: q6_load_at<12>(row, wd); break;
    default: q6_load_at<14>(row, wd); break;
    }
}

// ---------------------------------------------------------------- chunk bodies

// Accumulator update of one block/sub-block chain c with scale a.
template <int M, int NR0>
__device__ __forceinline__ void apply_scale(float2 (&acc)[NR0][M], const float2 (&c)[NR0][M],
                                            const float (&a)[NR0]) {
#pragma unroll
    for (int i = 0; i < NR0; ++i)
#pragma unroll
        for (int j = 0; j < M; ++j) acc[i][j] = fma2(make_float2(a[i], a[i]), c[i][j], acc[i][j]);
}

// Chain over 16 pairs with inputs x[j][0..31] (32 consecutive floats).
template <int M, int NR0>
__device__ __forceinline__ void chain32(float2 (&c)[NR0][M], const float2 (&w)[NR0][16], const float* xu,
                                        uint32_t xrs) {
#pragma unroll
    for (int i = 0; i < NR0; ++i)
#pragma unroll
        for (int j = 0; j < M; ++j) c[i][j] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        float4 xv[M];
#pragma unroll
        for (int j = 0; j < M; ++j) xv[j] = ldx4(xu + j * xrs + 4 * q);
#pragma unroll
        for (int i = 0; i < NR0; ++i)
#pragma unroll
            for (int j = 0; j < M; ++j) {
                c[i][j] = fma2(w[i][2 * q], make_float2(xv[j].x, xv[j].y), c[i][j]);
                c[i][j] = fma2(w[i][2 * q + 1], make_float2(xv[j].z, xv[j].w), c[i][j]);
            }
    }
}

template <int M, int NR0, bool FULL>
__device__ __forceinline__ void chunk_f16(const uint8_t* const (&rows)[NR0], const float* xc, uint32_t xrs,
                                          int nvals, float2 (&acc)[NR0][M]) {
    float2 c[NR0][M];
#pragma unroll
    for (int i = 0; i < NR0; ++i)
#pragma unroll
        for (int j = 0; j < M; ++j) c[i][j] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int g = 0; g < 17; ++g) {  // 8 values per step
        if (!FULL && 8 * g >= nvals) break;
        const bool second = FULL || (8 * g + 4 < nvals);
        float4 xa[M], xb[M];
#pragma unroll
        for (int j = 0; j < M; ++j) {
            xa[j] = ldx4(xc + j * xrs + 8 * g);
            xb[j] = second ? ldx4(xc + j * xrs + 8 * g + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < NR0; ++i) {
            const uint4 h = lds16(rows[i] + 16 * g);
            const float2 p0 = __half22float2(*reinterpret_cast<const __half2*>(&h.x));
            const float2 p1 = __half22float2(*reinterpret_cast<const __half2*>(&h.y));
            const float2 p2 = __half22float2(*reinterpret_cast<const __half2*>(&h.z));
            const float2 p3 = __half22float2(*reinterpret_cast<const __half2*>(&h.w));
#pragma unroll
            for (int j = 0; j < M; ++j) {
                c[i][j] = fma2(p0, make_float2(xa[j].x, xa[j].y), c[i][j]);
                c[i][j] = fma2(p1, make_float2(xa[j].z, xa[j].w), c[i][j]);
                if (second) {
                    c[i][j] = fma2(p2, make_float2(xb[j].x, xb[j].y), c[i][j]);
                    c[i][j] = fma2(p3, make_float2(xb[j].z, xb[j].w), c[i][j]);
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < NR0; ++i)
#pragma unroll
        for (int j = 0; j < M; ++j) acc[i][j] = add2(acc[i][j], c[i][j]);
}

template <int M, int NR0, bool FULL>
__device__ __forceinline__ void chunk_q8_0(const uint8_t* const (&rows)[NR0], const float* xc, uint32_t xrs,
                                           int nblk, float2 (&acc)[NR0][M]) {
    static_for<0, 8>([&](auto bc) {
        constexpr int B = decltype(bc)::value;
        if (!FULL && B >= nblk) return;
        float d[NR0];
        float2 w[NR0][16];
#pragma unroll
        for (int i = 0; i < NR0; ++i) dec_q8_0<B>(rows[i], d[i], w[i]);
        float2 c[NR0][M];
        chain32<M, NR0>(c, w, xc + 32 * B, xrs);
        apply_scale<M, NR0>(acc, c, d);
    });
}

template <int M, int NR0, bool FULL>
__device__ __forceinline__ void chunk_q5_0(const uint8_t* const (&rows)[NR0], const float* xc, uint32_t xrs,
                                           int nblk, float2 (&acc)[NR0][M]) {
    static_for<0, 8>([&](auto bc) {
        constexpr int B = decltype(bc)::value;
        if (!FULL && B >= nblk) return;
        float d[NR0];
        float2 w[NR0][16];
#pragma unroll
        for (int i = 0; i < NR0; ++i) dec_q5_0<B>(rows[i], d[i], w[i]);
        float2 c[NR0][M];
        chain32<M, NR0>(c, w, xc + 32 * B, xrs);
        apply_scale<M, NR0>(acc, c, d);
    });
}

// Q4_K super-block.  xs[u*M + j] = sum of the 32 inputs of sub-block u for
// input row j (computed once per chunk for the CTA, see xsum_q4_k).
template <int M, int NR0>
__device__ __forceinline__ void chunk_q4_k(const uint8_t* const (&rows)[NR0], const float* xc, uint32_t xrs,
                                           const float* xs, float2 (&acc)[NR0][M]) {
    float d[NR0], dmin[NR0];
    uint32_t s0[NR0], s1[NR0], s2[NR0];
#pragma unroll
    for (int i = 0; i < NR0; ++i) {
        const uint4 h = lds16(rows[i]);
        d[i] = h2f(h.x);
        dmin[i] = h2f(h.x >> 16);
        s0[i] = h.y;
        s1[i] = h.z;
        s2[i] = h.w;
    }
#pragma unroll
    for (int cq = 0; cq < 4; ++cq) {
        uint32_t q[NR0][8];
#pragma unroll
        for (int i = 0; i < NR0; ++i) {
            const uint4 a = lds16(rows[i] + 16 + 32 * cq), b = lds16(rows[i] + 32 + 32 * cq);
            q[i][0] = a.x; q[i][1] = a.y; q[i][2] = a.z; q[i][3] = a.w;
            q[i][4] = b.x; q[i][5] = b.y; q[i][6] = b.z; q[i][7] = b.w;
        }
#pragma unroll
        for (int H = 0; H < 2; ++H) {
            const int u = 2 * cq + H;
            float sc[NR0], mnv[NR0];
            float2 w[NR0][16];
#pragma unroll
            for (int i = 0; i < NR0; ++i) {
                uint32_t scu, mnu;
                q4k_scale_min(s0[i], s1[i], s2[i], u, scu, mnu);
                sc[i] = __fmul_rn(d[i], static_cast<float>(scu));
                mnv[i] = __fmul_rn(dmin[i], static_cast<float>(mnu));
                if (H == 0) dec_q4_k_sub<0>(q[i], w[i]); else dec_q4_k_sub<1>(q[i], w[i]);
            }
            float2 c[NR0][M];
            chain32<M, NR0>(c, w, xc + 32 * u, xrs);
            apply_scale<M, NR0>(acc, c, sc);
#pragma unroll
            for (int i = 0; i < NR0; ++i)
#pragma unroll
                for (int j = 0; j < M; ++j) acc[i][j].x = __fmaf_rn(-mnv[i], xs[u * M + j], acc[i][j].x);
        }
    }
}

// Sub-block input sums of one Q4_K chunk, per warp: lane (u = lane/4,
// quarter = lane%4) adds 8 inputs, then two xor-shuffles combine the quarters
// as (q0 + q1) + (q2 + q3).  The order is fixed and does not depend on M.
// xc is the staged [M][256] input slice.
template <int M>
__device__ __forceinline__ void xsum_q4_k(const float* xc, float* xs, int lane) {
    const int u = lane >> 2, qt = lane & 3;
#pragma unroll
    for (int j = 0; j < M; ++j) {
        const float4 a = ldx4(xc + j * 256 + 32 * u + 8 * qt);
        const float4 b = ldx4(xc + j * 256 + 32 * u + 8 * qt + 4);
        float s = __fadd_rn(__fadd_rn(__fadd_rn(a.x, a.y), __fadd_rn(a.z, a.w)),
                            __fadd_rn(__fadd_rn(b.x, b.y), __fadd_rn(b.z, b.w)));
        s = __fadd_rn(s, __shfl_xor_sync(0xFFFFFFFFu, s, 1));
        s = __fadd_rn(s, __shfl_xor_sync(0xFFFFFFFFu, s, 2));
        if (qt == 0) xs[u * M + j] = s;
    }
}

// Q6_K super-block staged at byte o of each row.
template <int M, int NR0>
__device__ __forceinline__ void chunk_q6_k(const uint8_t* const (&rows)[NR0], const float* xc, uint32_t xrs,
                                           int o, float2 (&acc)[NR0][M]) {
    uint32_t wd[NR0][53];
    float d[NR0];
#pragma unroll
    for (int i = 0; i < NR0; ++i) {
        q6_load(rows[i], o, wd[i]);
        d[i] = h2f(wd[i][52]);
    }
    const float2 bias = make_float2(-8388640.0f, -32800.0f);  // 2^23 + 32, 2^15 + 32
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int gh = 0; gh < 2; ++gh) {
                const int u = 8 * h + 2 * t + gh;  // sub-block of 16 values
                float a[NR0];
                float2 w[NR0][8];
#pragma unroll
                for (int i = 0; i < NR0; ++i) {
                    const int scb = static_cast<int>(static_cast<int8_t>((wd[i][48 + (u >> 2)] >> (8 * (u & 3))) & 0xFFu));
                    a[i] = __fmul_rn(d[i], static_cast<float>(scb));
#pragma unroll
                    for (int g4 = 0; g4 < 4; ++g4) {
                        const int g = 4 * gh + g4;
                        const uint32_t ql = wd[i][16 * h + 8 * (t & 1) + g];
                        const uint32_t qh = wd[i][32 + 8 * h + g];
                        const uint32_t lo = (t < 2 ? ql : (ql >> 4)) & 0x0F0F0F0Fu;
                        uint32_t hi;
                        if (t == 0) hi = (qh << 4) & 0x30303030u;
                        else if (t == 1) hi = (qh << 2) & 0x30303030u;
                        else if (t == 2) hi = qh & 0x30303030u;
                        else hi = (qh >> 2) & 0x30303030u;
                        const uint32_t v = lo | hi, v2 = v >> 16;
                        w[i][2 * g4] = add2(make_float2(fbits((v & 0xFFu) | 0x4B000000u), fbits((v & 0xFF00u) | 0x47000000u)), bias);
                        w[i][2 * g4 + 1] = add2(make_float2(fbits((v2 & 0xFFu) | 0x4B000000u), fbits((v2 & 0xFF00u) | 0x47000000u)), bias);
                    }
                }
                float2 c[NR0][M];
#pragma unroll
                for (int i = 0; i < NR0; ++i)
#pragma unroll
                    for (int j = 0; j < M; ++j) c[i][j] = make_float2(0.0f, 0.0f);
                const float* xu = xc + 128 * h + 32 * t + 16 * gh;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float4 xv[M];
#pragma unroll
                    for (int j = 0; j < M; ++j) xv[j] = ldx4(xu + j * xrs + 4 * q);
#pragma unroll
                    for (int i = 0; i < NR0; ++i)
#pragma unroll
                        for (int j = 0; j < M; ++j) {
                            c[i][j] = fma2(w[i][2 * q], make_float2(xv[j].x, xv[j].y), c[i][j]);
                            c[i][j] = fma2(w[i][2 * q + 1], make_float2(xv[j].z, xv[j].w), c[i][j]);
                        }
                }
                apply_scale<M, NR0>(acc, c, a);
            }
}

// ---------------------------------------------------------------- staging

// Fallback staging (the TMA path needs 16-byte aligned rows): copy chunk cc
// of one warp's rows with 2-byte loads into the positions a TMA box uses
// (W only needs 2-byte alignment).
template <int WT>
__device__ __forceinline__ void stage_w_plain(uint8_t* dst_rows, const uint8_t* wrow0, uint64_t row_bytes,
                                              int nrows, uint32_t cc, uint32_t k, int lane) {
    constexpr int BOX = Stage<WT>::kBox;
    uint32_t first, len;  // byte range of the chunk inside the row
    if constexpr (WT == kF16) {
        first = cc * 272u;
        len = 2u * min(136u, k - cc * 136u);
    } else if constexpr (WT == kQ8_0 || WT == kQ5_0) {
        constexpr uint32_t bb = (WT == kQ8_0) ? 34u : 22u;
        first = cc * 8u * bb;
        len = min(8u, k / 32u - cc * 8u) * bb;
    } else if constexpr (WT == kQ4_K) {
        first = cc * 144u;
        len = 144u;
    } else {
        first = cc * 210u;
        len = 210u;
    }
    const int so = Stage<WT>::sofs(cc);
    const uint32_t halves = len >> 1;
    for (int r = 0; r < nrows; ++r) {
        const uint16_t* src = reinterpret_cast<const uint16_t*>(wrow0 + static_cast<uint64_t>(r) * row_bytes + first);
        uint16_t* dst = reinterpret_cast<uint16_t*>(dst_rows + r * BOX + so);
        for (uint32_t h = lane; h < halves; h += 32) dst[h] = __ldg(src + h);
    }
}

// Fallback input staging: the [M][CV] slice of chunk cc, zero past k.
template <int M, int CV>
__device__ __forceinline__ void stage_x_plain(float* dst, const float* xb, uint32_t xrs, uint32_t cc, uint32_t k,
                                              int nthreads) {
    constexpr int Q = CV / 4;
    for (int idx = static_cast<int>(threadIdx.x); idx < M * Q; idx += nthreads) {
        const int j = idx / Q, q = idx - (idx / Q) * Q;
        const uint32_t col = cc * CV + 4u * q;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (col < k) v = ldg4(xb + static_cast<uint64_t>(j) * xrs + col);
        *reinterpret_cast<float4*>(dst + j * CV + 4 * q) = v;
    }
}

// ---------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync() {
    cluster_arrive();
    cluster_wait();
}

// f32 at the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ float ld_peer(const float* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// ---------------------------------------------------------------- per-chunk and per-row-block steps

// Decode + multiply one staged chunk for the warp's rows.
template <int WT, int M, int NR0>
__device__ __forceinline__ void mv_chunk(const uint8_t* st, uint32_t wstage, int warp, int lane, uint32_t cc,
                                         uint32_t k, float* xs, float2 (&acc)[NR0][M]) {
    constexpr int BOX = Stage<WT>::kBox;
    constexpr int CV = Stage<WT>::kValues;
    constexpr int ROWS = kLanes * NR0;
    const uint8_t* rows[NR0];
#pragma unroll
    for (int i = 0; i < NR0; ++i) rows[i] = st + (warp * ROWS + lane + 32 * i) * BOX;
    const float* xc = reinterpret_cast<const float*>(st + wstage);  // [M][CV]
    if constexpr (WT == kF16) {
        const int nv = static_cast<int>(min(136u, k - cc * 136u));
        if (nv == 136) chunk_f16<M, NR0, true>(rows, xc, CV, nv, acc);
        else chunk_f16<M, NR0, false>(rows, xc, CV, nv, acc);
    } else if constexpr (WT == kQ8_0 || WT == kQ5_0) {
        const int nb = static_cast<int>(min(8u, k / 32u - cc * 8u));
        if (nb == 8) {
            if constexpr (WT == kQ8_0) chunk_q8_0<M, NR0, true>(rows, xc, CV, nb, acc);
            else chunk_q5_0<M, NR0, true>(rows, xc, CV, nb, acc);
        } else {
            if constexpr (WT == kQ8_0) chunk_q8_0<M, NR0, false>(rows, xc, CV, nb, acc);
            else chunk_q5_0<M, NR0, false>(rows, xc, CV, nb, acc);
        }
    } else if constexpr (WT == kQ4_K) {
        xsum_q4_k<M>(xc, xs, lane);
        __syncwarp();
        chunk_q4_k<M, NR0>(rows, xc, CV, xs, acc);
    } else {
        chunk_q6_k<M, NR0>(rows, xc, CV, Stage<WT>::sofs(cc), acc);
    }
}

// End of a row block for one consumer warp: the range partial
// (acc.x + acc.y), then either the store (split 1) or the in-order sum of
// the cluster's ranges by rank 0.  Every thread of every CTA of the cluster
// reaches the cluster barrier once per row block.
template <int M, int NR0>
__device__ __forceinline__ void mv_finish(const float2 (&acc)[NR0][M], bool failed, const MvArgs& a, uint32_t b,
                                          uint32_t wrow0, bool wactive, bool consumer, int lane, int warp,
                                          uint32_t s, uint32_t S, uint32_t t, float* parts, uint32_t part_floats) {
    float part[NR0][M];
#pragma unroll
    for (int i = 0; i < NR0; ++i)
#pragma unroll
        for (int j = 0; j < M; ++j)
            part[i][j] = failed ? __int_as_float(0x7FC00000) : __fadd_rn(acc[i][j].x, acc[i][j].y);
    auto store = [&](int i, int j, float v) {
        const uint32_t row = wrow0 + static_cast<uint32_t>(lane + 32 * i);
        if (row < a.n) a.y[static_cast<uint64_t>(b) * a.ybs + static_cast<uint64_t>(j) * a.yrs + row] = v;
    };
    if (S == 1) {
        if (wactive) {
#pragma unroll
            for (int i = 0; i < NR0; ++i)
#pragma unroll
                for (int j = 0; j < M; ++j) store(i, j, part[i][j]);
        }
        return;
    }
    float* buf = parts + (t & 1u) * part_floats;
    if (s != 0 && consumer) {
#pragma unroll
        for (int i = 0; i < NR0; ++i)
#pragma unroll
            for (int j = 0; j < M; ++j) buf[((warp * NR0 + i) * M + j) * 32 + lane] = part[i][j];
    }
    cluster_sync();  // phase t: the ranges' partials of this row block are published
    if (s == 0 && wactive) {
#pragma unroll
        for (int i = 0; i < NR0; ++i)
#pragma unroll
            for (int j = 0; j < M; ++j) {
                const float* slot = buf + ((warp * NR0 + i) * M + j) * 32 + lane;
                float v = part[i][j];
                for (uint32_t r = 1; r < S; ++r) v = __fadd_rn(v, ld_peer(slot, r));
                store(i, j, v);
            }
    }
}

// ---------------------------------------------------------------- the kernel

// Persistent kernel.  A cluster of `split` CTAs walks the row blocks
// cid, cid + nclusters, ... (a row block is G row groups of ROWS = 32*NR0
// rows of one batch); CTA rank s of the cluster handles K range s of every
// row block.  A CTA has G consumer warps (one row group each) and one
// producer warp.  Each pipeline stage holds one TMA box of the row block's
// rows (G*ROWS x BOX bytes) and one box of the matching inputs (M x CV
// floats).  The producer fills a stage once all consumer warps released it
// (mbarrier `empty`, G arrivals) and runs on into the next row block;
// consumers wait for the bytes (mbarrier `full`) and release each stage as
// soon as they are done with it.  After a row block, CTAs of rank > 0 leave
// their partial sums in shared memory (double-buffered by row-block parity),
// one cluster barrier publishes them, and rank 0 adds them in range order
// through distributed shared memory and stores y.  The producer takes part in
// that barrier split-phase (arrive after issuing a row block, wait one row
// block later), so it never stalls the stream.
template <int WT, int M, int NR0>
__global__ void __launch_bounds__((kMaxWarps + 1) * 32)
rem_mv_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap, const MvArgs a) {
    constexpr int BOX = Stage<WT>::kBox;
    constexpr int CV = Stage<WT>::kValues;
    constexpr int ROWS = kLanes * NR0;
    constexpr uint32_t XBYTES = M * CV * 4;
    constexpr uint32_t XPAD = (XBYTES + 127u) & ~127u;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = static_cast<int>(blockDim.x >> 5) - 1;  // consumer warps; warp G produces
    const bool producer = warp == G;
    const uint32_t S = a.split;
    const int D = static_cast<int>(a.stages);
    const uint32_t s = S > 1 ? cluster_rank() : 0u;
    const uint32_t cid = blockIdx.x / S;
    const uint32_t ncl = gridDim.x / S;
    const uint32_t wstage = static_cast<uint32_t>(G * ROWS * BOX);
    const uint32_t stage_bytes = wstage + XPAD;
    const uint32_t part_floats = static_cast<uint32_t>(G * NR0 * M * 32);
    float* parts = reinterpret_cast<float*>(smem + D * stage_bytes);  // [2][G][NR0][M][32] when S > 1
    uint64_t* full = reinterpret_cast<uint64_t*>(parts + (S > 1 ? 2 * part_floats : 0));
    uint64_t* empty = full + kMaxStages;
    float* xs = reinterpret_cast<float*>(empty + kMaxStages) + warp * (8 * kMaxRows);
    const uint32_t c0 = static_cast<uint32_t>((static_cast<uint64_t>(s) * a.nchunk) / S);
    const uint32_t c1 = static_cast<uint32_t>((static_cast<uint64_t>(s + 1) * a.nchunk) / S);
    const int nck = static_cast<int>(c1 - c0);
    const uint32_t nblocks = a.cpb * a.batch;  // row blocks of the whole launch

    // row block -> (batch, first row in the batch)
    auto block_origin = [&](uint32_t rb, uint32_t& b, uint32_t& row0) {
        b = rb / a.cpb;
        row0 = (rb - b * a.cpb) * static_cast<uint32_t>(G * ROWS);
    };

    bool failed = false;

    if (!a.aligned) {
        // ---- plain staging: every warp copies, consumers compute, one stage
        const int nthreads = static_cast<int>(blockDim.x);
        for (uint32_t rb = cid, t = 0; rb < nblocks; rb += ncl, ++t) {
            uint32_t b, row0;
            block_origin(rb, b, row0);
            const uint32_t wrow0 = row0 + static_cast<uint32_t>(warp * ROWS);
            const bool wactive = !producer && wrow0 < a.n;
            const float* xb = a.x + static_cast<uint64_t>(b) * a.xbs;
            const int wrows = wactive ? static_cast<int>(min(static_cast<uint32_t>(ROWS), a.n - wrow0)) : 0;
            const uint8_t* wrow_ptr = a.w + (static_cast<uint64_t>(b) * a.n + wrow0) * a.row_bytes;
            float2 acc[NR0][M];
#pragma unroll
            for (int i = 0; i < NR0; ++i)
#pragma unroll
                for (int j = 0; j < M; ++j) acc[i][j] = make_float2(0.0f, 0.0f);
            for (int i = 0; i < nck; ++i) {
                const uint32_t cc = c0 + static_cast<uint32_t>(i);
                if (wactive) stage_w_plain<WT>(smem + warp * ROWS * BOX, wrow_ptr, a.row_bytes, wrows, cc, a.k, lane);
                stage_x_plain<M, CV>(reinterpret_cast<float*>(smem + wstage), xb, a.xrs, cc, a.k, nthreads);
                __syncthreads();
                if (wactive) mv_chunk<WT, M, NR0>(smem, wstage, warp, lane, cc, a.k, xs, acc);
                __syncthreads();
            }
            mv_finish<M, NR0>(acc, false, a, b, wrow0, wactive, !producer, lane, warp, s, S, t, parts, part_floats);
        }
        if (S > 1) cluster_sync();  // no CTA leaves while a peer may still read it
        return;
    }

    // ---- TMA pipeline
    const uint32_t fb = smem_u32(full), eb = smem_u32(empty);
    if (threadIdx.x == 0) {
        for (int t = 0; t < D; ++t) {
            mbar_init(fb + 8 * t, 1);
            mbar_init(eb + 8 * t, static_cast<uint32_t>(G));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (producer) {
        uint32_t i = 0;  // running chunk counter over all row blocks
        bool stop = false;
        uint32_t t = 0;
        for (uint32_t rb = cid; rb < nblocks; rb += ncl, ++t) {
            uint32_t b, row0;
            block_origin(rb, b, row0);
            const uint64_t grow0 = static_cast<uint64_t>(b) * a.n + row0;
            if (lane == 0 && !stop) {
                for (int q = 0; q < nck; ++q, ++i) {
                    const int st = static_cast<int>(i % D);
                    if (i >= static_cast<uint32_t>(D) &&
                        !mbar_wait(eb + 8 * st, static_cast<uint32_t>((i / D - 1) & 1))) {
                        stop = true;
                        break;
                    }
                    const uint32_t cc = c0 + static_cast<uint32_t>(q);
                    uint8_t* sp = smem + st * stage_bytes;
                    mbar_expect_tx(fb + 8 * st, wstage + XBYTES);
                    tma_load_2d(smem_u32(sp), &wmap, static_cast<int32_t>(Stage<WT>::gofs(cc) / 2),
                                static_cast<int32_t>(grow0), fb + 8 * st);
                    tma_load_3d(smem_u32(sp + wstage), &xmap, static_cast<int32_t>(cc * CV),
                                a.x_bm ? static_cast<int32_t>(b) : 0, a.x_bm ? 0 : static_cast<int32_t>(b),
                                fb + 8 * st);
                }
            }
            __syncwarp();
            if (S > 1) {
                if (t > 0) cluster_wait();  // phase t-1
                cluster_arrive();            // phase t
            }
        }
        if (S > 1 && t > 0) cluster_wait();
        // every copy issued has landed before the CTA can exit (bounded)
        if (lane == 0) {
            const uint32_t issued = i;
            for (uint32_t r = issued > static_cast<uint32_t>(D) ? issued - D : 0u; r < issued; ++r)
                (void)mbar_wait(fb + 8 * (r % D), static_cast<uint32_t>((r / D) & 1));
        }
        __syncwarp();
        if (S > 1) cluster_sync();
        return;
    }

    uint32_t i = 0;
    for (uint32_t rb = cid, t = 0; rb < nblocks; rb += ncl, ++t) {
        uint32_t b, row0;
        block_origin(rb, b, row0);
        const uint32_t wrow0 = row0 + static_cast<uint32_t>(warp * ROWS);
        const bool wactive = wrow0 < a.n;
        float2 acc[NR0][M];
#pragma unroll
        for (int r = 0; r < NR0; ++r)
#pragma unroll
            for (int j = 0; j < M; ++j) acc[r][j] = make_float2(0.0f, 0.0f);
        for (int q = 0; q < nck; ++q, ++i) {
            const int st = static_cast<int>(i % D);
            if (!failed &&
                !__all_sync(0xFFFFFFFFu, mbar_wait(fb + 8 * st, static_cast<uint32_t>((i / D) & 1))))
                failed = true;
            if (failed) continue;  // keep walking so every barrier below is still reached
            if (wactive)
                mv_chunk<WT, M, NR0>(smem + st * stage_bytes, wstage, warp, lane, c0 + static_cast<uint32_t>(q), a.k,
                                     xs, acc);
            __syncwarp();
            if (lane == 0) mbar_arrive(eb + 8 * st);
        }
        mv_finish<M, NR0>(acc, failed, a, b, wrow0, wactive, true, lane, warp, s, S, t, parts, part_floats);
    }
    if (S > 1) cluster_sync();
}

}  // namespace dev
}  // namespace rem

// Each translation unit instantiates four M values of one weight format,
// both NR0, and exposes them through a lookup function.
#define REM_K(WT, M) \
    {(const void*)&::rem::dev::rem_mv_kernel<WT, M, 1>, (const void*)&::rem::dev::rem_mv_kernel<WT, M, 2>}
#define REM_INSTANTIATE4(WT, NAME, M0)                                                             \
    namespace rem {                                                                                \
    const void* NAME(int m, int nr0) {                                                             \
        static const void* const table[4][2] = {REM_K(WT, M0), REM_K(WT, M0 + 1), REM_K(WT, M0 + 2), \
                                                REM_K(WT, M0 + 3)};                                \
        if (m < M0 || m > M0 + 3 || nr0 < 1 || nr0 > 2) return nullptr;                           \
        return table[m - M0][nr0 - 1];                                                             \
    }                                                                                              \
    }
