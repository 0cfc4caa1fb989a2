// rem_mv.cuh -- the row-exact few-row mat-vec kernel for sm_103a.
//
// y[b, j, i] = sum_k W[b*n + i, k] * x[b, j, k],  j < M <= 8
// (mlx-native 0.18.0 src/ops/row_exact_matvec.rs, module doc).
//
// Work mapping.  A warp owns 32*NR0 consecutive weight rows.  Its lanes form
// H groups (H = 1: lane l holds rows l and, with NR0 = 2, l+32 for all M
// input rows; H = 2: lanes l and l+16 both hold rows l and l+16 (and, with
// NR0 = 2, l+32 and l+48), for the first and the second half of the input
// rows).  All lanes of a warp work on
// the same K positions at the same time, so every input load is a
// shared-memory broadcast (one address per lane group) feeding NR0*H rows,
// and every weight row is read from HBM exactly once for all M input rows.  K is cut into `split` contiguous ranges of chunks.  The
// `split` CTAs of a thread-block cluster share the same rows and take one
// range each; their partial sums are added in range order through
// distributed shared memory (each output by one rank of the cluster).  Each
// CTA streams its chunks through a ring of TMA stages: one box of weight rows
// and one box of the matching inputs per stage, completed on one mbarrier.
//
// Row exactness (module doc "Row exactness").  The arithmetic of output
// (i, j) depends only on row i's bytes, input row j and `split`:
//   * each block / sub-block u contributes through one packed chain
//     c = fma2(w[2p..2p+1], x[2p..2p+1], c) over its value pairs in order,
//   * then acc = fma2((a_u, a_u), c, acc) with the block scale a_u
//     (Q4_K also acc.x = fma(-min_u, sum(x of u), acc.x), affine groups
//     acc.x = fma(bias_u, sum(x of u), acc.x); F16 / BF16 / F32 chunks
//     acc = acc + c),
//   * a range's partial is acc.x + acc.y, and ranges are summed in order;
//   * an optional epilogue y = fma(alpha, partial sum, beta * c) per output.
// Nothing in that sequence depends on M, NR0, H, the CTA packing or the
// staging path, so row j of an M-row launch equals the same row of an M=1
// launch bit for bit.  fma.rn.f32x2 performs two independent, correctly
// rounded FMAs, identical to two scalar fmaf.
//
// Block decode.  Integer codes become exact floats without a conversion
// instruction: a code q placed in mantissa bits [p, p+w) under the exponent
// 2^(23-p) reads as 2^(23-p) + q, and one add of -(2^(23-p) + offset)
// yields q - offset exactly (offset 128 for int8 stored as uint8, 16 for
// Q5_0, 32 for Q6_K, 0 for Q4_K and affine codes).
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

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier / TMA

// Weight bytes a CTA prefetches into L2 ahead of its dependency wait.
constexpr uint32_t kPrefetchBytes = 64u << 10;

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

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait: true once the phase of `parity` has completed, false when it
// has not completed `limit_ns` nanoseconds (of the global timer) after the
// first unsuccessful try.  The poll count is capped as well, so the wait
// ends even if the timer were not to advance.
// One non-blocking test of the phase of `parity` (mbarrier.test_wait, acquire
// when it reports the phase complete).  Issued ahead of the point where the
// answer is needed, its latency overlaps other work.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 0; it < (1u << 26); ++it) {
#pragma unroll 1
        for (int i = 0; i < 8; ++i)
            if (mbar_try(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// A wait ran out: record it in the launch's status word (read back by
// rem_device_status) before the caller writes NaN where its results go.
__device__ __forceinline__ void report_timeout(uint32_t* status, uint32_t what) {
    if (status) atomicOr(status, what);
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

// Prefetch one TMA box of weights into L2 (no shared-memory destination, no
// completion to wait for).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// Programmatic dependent launch: let the next kernel of the stream start its
// prologue, and wait until every kernel this one depends on has completed
// and its writes are visible (returns at once without such a dependency).
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- format traits

// Staged bytes per row (the TMA box width) and the byte position inside the
// staged row where chunk `cc` starts.
// Affine codes (the primary template): chunk cc is the kBytes bytes at
// kBytes*cc -- 128 bytes of 4- or 8-bit codes (256 / 128 values) staged as a
// 144-byte window, or 256 codes of 3, 5 or 6 bits (96, 160, 192 bytes)
// staged as 112-, 176- or 208-byte windows (an odd number of 16-byte units
// keeps the 32 lanes' reads on distinct bank quads).
template <int WT> struct Stage {
    static_assert(is_affine(WT), "no staging geometry for this weight type");
    static constexpr int kValues = chunk_values(WT), kBox = chunk_box(WT);
    static constexpr uint32_t kBytes = static_cast<uint32_t>(kValues * affine_bits(WT) / 8);
    static_assert(kBytes % 16 == 0 && kBytes <= static_cast<uint32_t>(kBox), "chunk bytes");
    __device__ static uint32_t gofs(uint32_t cc) { return cc * kBytes; }
    __device__ static int sofs(uint32_t) { return 0; }
};
template <> struct Stage<kF16> {
    static constexpr int kValues = 72, kBox = 144;
    __device__ static uint32_t gofs(uint32_t cc) { return cc * 144u; }  // global byte offset of the box
    __device__ static int sofs(uint32_t) { return 0; }
};
template <> struct Stage<kBF16> {
    static constexpr int kValues = 72, kBox = 144;
    __device__ static uint32_t gofs(uint32_t cc) { return cc * 144u; }
    __device__ static int sofs(uint32_t) { return 0; }
};
template <> struct Stage<kF32> {
    static constexpr int kValues = 36, kBox = 144;
    __device__ static uint32_t gofs(uint32_t cc) { return cc * 144u; }
    __device__ static int sofs(uint32_t) { return 0; }
};
// Q8_0 chunks are 4 blocks (136 B): stage the 16-byte aligned 144-byte
// window that contains them; they start 0 or 8 bytes into it.
template <> struct Stage<kQ8_0> {
    static constexpr int kValues = 128, kBox = 144;
    __device__ static uint32_t gofs(uint32_t cc) { return (cc * 136u) & ~15u; }
    __device__ static int sofs(uint32_t cc) { return static_cast<int>((cc * 136u) & 15u); }
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

// lop3: (a & b) | c
__device__ __forceinline__ uint32_t lop_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// lop3: bitwise b ? (a ^ c) : c -- the bits of a under mask b with c's bits
// flipped, c elsewhere
__device__ __forceinline__ uint32_t lop_sel_xor(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// lop3: bitwise c ? a : b
__device__ __forceinline__ uint32_t lop_sel(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xE4;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Bytes 0 and 1 of v as two exact floats: the bits under masks m0 (within
// bits 0..7) and m1 (within bits 8..15) become mantissa bits under the
// exponents 2^23 and 2^15, then `bias` removes 2^23 (2^15) and the code offset.
__device__ __forceinline__ float2 bytes01_u(uint32_t v, uint32_t m0, uint32_t m1, float2 bias) {
    return add2(make_float2(fbits(lop_and_or(v, m0, 0x4B000000u)), fbits(lop_and_or(v, m1, 0x47000000u))), bias);
}
// Bytes 0 and 1 of v read as int8: the sign bit is flipped on the way in
// (q + 128 in 0..255), and the bias removes 2^23 + 128 (2^15 + 128).
__device__ __forceinline__ float2 bytes01_s(uint32_t v) {
    return add2(make_float2(fbits(lop_sel_xor(v, 0xFFu, 0x4B000080u)), fbits(lop_sel_xor(v, 0xFF00u, 0x47008000u))),
                make_float2(-8388736.0f, -32896.0f));
}

// Byte b (0..3) of w, masked to `mask` (0x3F or 0xFF), as an exact float.
template <int B>
__device__ __forceinline__ float ubyte_f(uint32_t w, uint32_t mask) {
    const uint32_t v = B >= 2 ? (w >> 16) : w;
    if constexpr ((B & 1) == 0) return fbits(lop_and_or(v, mask, 0x4B000000u)) - 8388608.0f;
    else return fbits(lop_and_or(v, mask << 8, 0x47000000u)) - 32768.0f;
}
// Byte b (0..3) of w read as int8, as an exact float.
template <int B>
__device__ __forceinline__ float sbyte_f(uint32_t w) {
    const uint32_t v = B >= 2 ? (w >> 16) : w;
    if constexpr ((B & 1) == 0) return fbits(lop_sel_xor(v, 0xFFu, 0x4B000080u)) - 8388736.0f;
    else return fbits(lop_sel_xor(v, 0xFF00u, 0x47008000u)) - 32896.0f;
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

// Word I (0..3) of a 16-byte line.
template <int I>
__device__ __forceinline__ uint32_t word_of(const uint4& v) {
    if constexpr (I == 0) return v.x;
    else if constexpr (I == 1) return v.y;
    else if constexpr (I == 2) return v.z;
    else return v.w;
}

// Spread the 4 low bits of h to bit 4 of each byte (bit k -> bit 8k+4).
__device__ __forceinline__ uint32_t spread4(uint32_t h) { return (h * 0x02040810u) & 0x10101010u; }

// A 32-value block of a staged chunk: load() takes its bytes from shared
// memory, group<Q>() yields values 4Q..4Q+3 as two pairs (decoded when the
// chain needs them, so only the block's raw words stay in registers).
//
// Q8_0 block at byte POS (even) of a 16-aligned staged row; d, then 32 int8.
template <int POS>
struct BlkQ8 {
    static constexpr int off = POS, p0 = off >> 4, bo = off & 15;
    uint32_t W[12];
    float d;
    __device__ __forceinline__ void load(const uint8_t* row) {
        const uint4 v0 = lds16(row + 16 * p0), v1 = lds16(row + 16 * (p0 + 1)), v2 = lds16(row + 16 * (p0 + 2));
        W[0] = v0.x; W[1] = v0.y; W[2] = v0.z; W[3] = v0.w;
        W[4] = v1.x; W[5] = v1.y; W[6] = v1.z; W[7] = v1.w;
        W[8] = v2.x; W[9] = v2.y; W[10] = v2.z; W[11] = v2.w;
        const uint32_t dw = W[bo >> 2];
        d = h2f((bo & 2) ? (dw >> 16) : dw);
    }
    template <int Q>
    __device__ __forceinline__ void group(float2& w01, float2& w23) const {
        const uint32_t v = u32_at<bo + 2 + 4 * Q>(W);
        w01 = bytes01_s(v);
        w23 = bytes01_s(v >> 16);
    }
};

// Q5_0 block at byte POS (even): d, qh (bit e = bit 4 of element e), then
// 16 bytes whose low nibbles are elements 0..15 and high nibbles 16..31.
template <int POS>
struct BlkQ5 {
    static constexpr int off = POS, p0 = off >> 4, bo = off & 15;
    uint32_t qs[4];
    uint32_t qh;
    float d;
    __device__ __forceinline__ void load(const uint8_t* row) {
        const uint4 v0 = lds16(row + 16 * p0), v1 = lds16(row + 16 * (p0 + 1));
        uint4 v2 = make_uint4(0u, 0u, 0u, 0u);
        if constexpr (bo + 22 > 32) v2 = lds16(row + 16 * (p0 + 2));
        const uint32_t W[12] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w, v2.x, v2.y, v2.z, v2.w};
        const uint32_t dw = W[bo >> 2];
        d = h2f((bo & 2) ? (dw >> 16) : dw);
        qh = u32_at<bo + 2>(W);
        qs[0] = u32_at<bo + 6>(W);
        qs[1] = u32_at<bo + 10>(W);
        qs[2] = u32_at<bo + 14>(W);
        qs[3] = u32_at<bo + 18>(W);
    }
    template <int Q>
    __device__ __forceinline__ void group(float2& w01, float2& w23) const {
        const uint32_t nib = Q < 4 ? qs[Q & 3] : (qs[Q & 3] >> 4);
        const uint32_t v = lop_and_or(nib, 0x0F0F0F0Fu, spread4((qh >> (4 * Q)) & 0xFu));
        const float2 bias = make_float2(-8388624.0f, -32784.0f);  // 2^23 + 16, 2^15 + 16
        w01 = bytes01_u(v, 0xFFu, 0xFF00u, bias);
        w23 = bytes01_u(v >> 16, 0xFFu, 0xFF00u, bias);
    }
};

// Q4_K: values 4Q..4Q+3 of sub-block 2c+H from qs word v = bytes 4Q..4Q+3
// of the chunk's 32 bytes.  Low nibbles (H = 0) sit at bits 0, 8, 16, 24;
// high nibbles (H = 1) at 4, 12, 20, 28.  A nibble at bit p is read under
// the exponent 2^(23-p); bits 20..31 go through v >> 12 first.
template <int H>
__device__ __forceinline__ void q4k_group(uint32_t v, float2& w01, float2& w23) {
    const uint32_t s = v >> 12;
    if constexpr (H == 0) {
        w01 = add2(make_float2(fbits(lop_and_or(v, 0xFu, 0x4B000000u)), fbits(lop_and_or(v, 0xF00u, 0x47000000u))),
                   make_float2(-8388608.0f, -32768.0f));
        w23 = add2(make_float2(fbits(lop_and_or(v, 0xF0000u, 0x43000000u)), fbits(lop_and_or(s, 0xF000u, 0x45000000u))),
                   make_float2(-128.0f, -2048.0f));
    } else {
        w01 = add2(make_float2(fbits(lop_and_or(v, 0xF0u, 0x49000000u)), fbits(lop_and_or(v, 0xF000u, 0x45000000u))),
                   make_float2(-524288.0f, -2048.0f));
        w23 = add2(make_float2(fbits(lop_and_or(s, 0xF00u, 0x47000000u)), fbits(lop_and_or(s, 0xF0000u, 0x43000000u))),
                   make_float2(-32768.0f, -128.0f));
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

// Q6_K: values l = 4G..4G+3 of quarter T of half H (elements 128H + 32T + l).
// Low nibbles come from ql word 16H + 8(T&1) + G (the low nibble for T < 2,
// the high one for T >= 2), the two high bits from bits 2T, 2T+1 of qh word
// 32 + 8H + G; one select puts them at bits 4..5 of each byte, and the 0x3F
// masks drop the unused bits 6..7.
template <int H, int T, int G>
__device__ __forceinline__ void q6k_group(const uint32_t (&wd)[53], float2& w01, float2& w23) {
    const uint32_t ql = wd[16 * H + 8 * (T & 1) + G];
    const uint32_t qh = wd[32 + 8 * H + G];
    const uint32_t lo = T < 2 ? ql : (ql >> 4);
    const uint32_t hi = T == 0 ? (qh << 4) : T == 1 ? (qh << 2) : T == 2 ? qh : (qh >> 2);
    const uint32_t v = lop_sel(lo, hi, 0x0F0F0F0Fu);
    const float2 bias = make_float2(-8388640.0f, -32800.0f);  // 2^23 + 32, 2^15 + 32
    w01 = bytes01_u(v, 0x3Fu, 0x3F00u, bias);
    w23 = bytes01_u(v >> 16, 0x3Fu, 0x3F00u, bias);
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

// The chain of one block / sub-block of 4*NG values: for each group Q of 4
// values, gen(Q, i, w01, w23) yields row i's values 4Q..4Q+3 and the chain
// takes c = fma2(w01, x[4Q..4Q+1], c), c = fma2(w23, x[4Q+2..4Q+3], c).
// Input row j of the group sits at xu + j*XS + 4Q in shared memory.  Only the
// group's decoded values and one input quad are live at a time.
template <int M, int NR0, int NG, int XS, typename Gen>
__device__ __forceinline__ void chain(float2 (&c)[NR0][M], const float* xu, Gen&& gen) {
#pragma unroll
    for (int i = 0; i < NR0; ++i)
#pragma unroll
        for (int j = 0; j < M; ++j) c[i][j] = make_float2(0.0f, 0.0f);
    static_for<0, NG>([&](auto qc) {
        constexpr int Q = decltype(qc)::value;
        float2 w01[NR0], w23[NR0];
#pragma unroll
        for (int i = 0; i < NR0; ++i) gen(qc, i, w01[i], w23[i]);
#pragma unroll
        for (int j = 0; j < M; ++j) {
            const float4 xv = ldx4(xu + j * XS + 4 * Q);
#pragma unroll
            for (int i = 0; i < NR0; ++i) {
                c[i][j] = fma2(w01[i], make_float2(xv.x, xv.y), c[i][j]);
                c[i][j] = fma2(w23[i], make_float2(xv.z, xv.w), c[i][j]);
            }
        }
    });
}

// The same walk over groups of 4 values, accumulating straight into acc
// (acc = fma2(w01, x[4Q..4Q+1], acc), acc = fma2(w23, x[4Q+2..4Q+3], acc)):
// for weights whose values gen() already dequantizes element by element.
template <int M, int NR0, int NG, int XS, typename Gen>
__device__ __forceinline__ void chain_acc(float2 (&acc)[NR0][M], const float* xu, Gen&& gen) {
    static_for<0, NG>([&](auto qc) {
        constexpr int Q = decltype(qc)::value;
        float2 w01[NR0], w23[NR0];
#pragma unroll
        for (int i = 0; i < NR0; ++i) gen(qc, i, w01[i], w23[i]);
#pragma unroll
        for (int j = 0; j < M; ++j) {
            const float4 xv = ldx4(xu + j * XS + 4 * Q);
#pragma unroll
            for (int i = 0; i < NR0; ++i) {
                acc[i][j] = fma2(w01[i], make_float2(xv.x, xv.y), acc[i][j]);
                acc[i][j] = fma2(w23[i], make_float2(xv.z, xv.w), acc[i][j]);
            }
        }
    });
}

// F16 chunk of 72 values (a zero-filled tail past k adds exact zeros).
template <int M, int NR0>
__device__ __forceinline__ void chunk_f16(const uint8_t* const (&rows)[NR0], const float* xc,
                                          float2 (&acc)[NR0][M]) {
    float2 c[NR0][M];
#pragma unroll
    for (int i = 0; i < NR0; ++i)
#pragma unroll
        for (int j = 0; j < M; ++j) c[i][j] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int g = 0; g < 9; ++g) {  // 8 values per step
        float2 p[NR0][4];
#pragma unroll
        for (int i = 0; i < NR0; ++i) {
            const uint4 h = lds16(rows[i] + 16 * g);
            p[i][0] = __half22float2(*reinterpret_cast<const __half2*>(&h.x));
            p[i][1] = __half22float2(*reinterpret_cast<const __half2*>(&h.y));
            p[i][2] = __half22float2(*reinterpret_cast<const __half2*>(&h.z));
            p[i][3] = __half22float2(*reinterpret_cast<const __half2*>(&h.w));
        }
#pragma unroll
        for (int j = 0; j < M; ++j) {
            const float4 xa = ldx4(xc + j * 72 + 8 * g);
            const float4 xb = ldx4(xc + j * 72 + 8 * g + 4);
#pragma unroll
            for (int i = 0; i < NR0; ++i) {
                c[i][j] = fma2(p[i][0], make_float2(xa.x, xa.y), c[i][j]);
                c[i][j] = fma2(p[i][1], make_float2(xa.z, xa.w), c[i][j]);
                c[i][j] = fma2(p[i][2], make_float2(xb.x, xb.y), c[i][j]);
                c[i][j] = fma2(p[i][3], make_float2(xb.z, xb.w), c[i][j]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < NR0; ++i)
#pragma unroll
        for (int j = 0; j < M; ++j) acc[i][j] = add2(acc[i][j], c[i][j]);
}

// BF16 pair from a 32-bit word: the two halves are the upper 16 bits of
// binary32 values (exact).
__device__ __forceinline__ float2 bf16x2(uint32_t v) { return make_float2(fbits(v << 16), fbits(v & 0xFFFF0000u)); }

// BF16 chunk of 72 values, F32 chunk of 36 values: the same chain as F16
// (pairs in order, then acc = acc + c per chunk).
template <int M, int NR0, int WT>
__device__ __forceinline__ void chunk_dense(const uint8_t* const (&rows)[NR0], const float* xc,
                                            float2 (&acc)[NR0][M]) {
    constexpr int CV = Stage<WT>::kValues;
    constexpr int PER = WT == kF32 ? 4 : 8;  // values per 16-byte load
    float2 c[NR0][M];
#pragma unroll
    for (int i = 0; i < NR0; ++i)
#pragma unroll
        for (int j = 0; j < M; ++j) c[i][j] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int g = 0; g < CV / PER; ++g) {
        float2 p[NR0][PER / 2];
#pragma unroll
        for (int i = 0; i < NR0; ++i) {
            const uint4 h = lds16(rows[i] + 16 * g);
            if constexpr (WT == kF32) {
                p[i][0] = make_float2(fbits(h.x), fbits(h.y));
                p[i][1] = make_float2(fbits(h.z), fbits(h.w));
            } else {
                p[i][0] = bf16x2(h.x);
                p[i][1] = bf16x2(h.y);
                p[i][2] = bf16x2(h.z);
                p[i][3] = bf16x2(h.w);
            }
        }
#pragma unroll
        for (int j = 0; j < M; ++j) {
#pragma unroll
            for (int q = 0; q < PER / 4; ++q) {
                const float4 xv = ldx4(xc + j * CV + PER * g + 4 * q);
#pragma unroll
                for (int i = 0; i < NR0; ++i) {
                    c[i][j] = fma2(p[i][2 * q], make_float2(xv.x, xv.y), c[i][j]);
                    c[i][j] = fma2(p[i][2 * q + 1], make_float2(xv.z, xv.w), c[i][j]);
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < NR0; ++i)
#pragma unroll
        for (int j = 0; j < M; ++j) acc[i][j] = add2(acc[i][j], c[i][j]);
}

// NB 32-value blocks (Q8_0 or Q5_0) of one staged chunk, block b at byte
// O + STRIDE*b of each staged row.  Blocks past k are zero-filled (scale 0,
// inputs 0) and add exact zeros.
template <int M, int NR0, template <int> class Blk, int NB, int STRIDE, int O>
__device__ __forceinline__ void chunk_blocks32(const uint8_t* const (&rows)[NR0], const float* xc,
                                               float2 (&acc)[NR0][M]) {
    constexpr int CV = 32 * NB;
    static_for<0, NB>([&](auto bc) {
        constexpr int B = decltype(bc)::value;
        Blk<O + STRIDE * B> blk[NR0];
        float d[NR0];
#pragma unroll
        for (int i = 0; i < NR0; ++i) {
            blk[i].load(rows[i]);
            d[i] = blk[i].d;
        }
        float2 c[NR0][M];
        chain<M, NR0, 8, CV>(c, xc + 32 * B, [&](auto qc, int i, float2& w01, float2& w23) {
            blk[i].template group<decltype(qc)::value>(w01, w23);
        });
        apply_scale<M, NR0>(acc, c, d);
    });
}

// Q4_K super-block.  Every weight is dequantized on its own, as the format
// defines it: w = fl(fl(d*sc)*q) - fl(dmin*mn).  d*sc (a binary16 times a
// 6-bit integer) and d*sc*q (times a 4-bit code) are exact in binary32, so
// the definition is one rounding of a*q - b, which is fma(a, q, -b) bit for
// bit.  Then acc += w*x.  (Folding the min into a sum of the inputs, a*sum(q*x)
// - b*sum(x), would round the two large terms separately and lose the
// accuracy of a weight that is their small difference.)
// Sub-block scales and mins: s < 4 from bytes s of scales[0..3] / [4..7];
// s >= 4 joins the low (high) nibble of scales[s+4] with the top two bits of
// scales[s-4] (scales[s]) -- one select per word.
template <int M, int NR0>
__device__ __forceinline__ void chunk_q4_k(const uint8_t* const (&rows)[NR0], const float* xc,
                                           float2 (&acc)[NR0][M]) {
    float d[NR0], dmin[NR0];
    uint32_t scw[NR0][2], mnw[NR0][2];
#pragma unroll
    for (int i = 0; i < NR0; ++i) {
        const uint4 h = lds16(rows[i]);
        d[i] = h2f(h.x);
        dmin[i] = h2f(h.x >> 16);
        scw[i][0] = h.y;
        mnw[i][0] = h.z;
        scw[i][1] = lop_sel(h.w, h.y >> 2, 0x0F0F0F0Fu);
        mnw[i][1] = lop_sel(h.w >> 4, h.z >> 2, 0x0F0F0F0Fu);
    }
    static_for<0, 4>([&](auto cqc) {
        constexpr int cq = decltype(cqc)::value;
        static_for<0, 2>([&](auto hc) {
            constexpr int H = decltype(hc)::value;
            constexpr int u = 2 * cq + H;
            float2 a2[NR0], nb2[NR0];
#pragma unroll
            for (int i = 0; i < NR0; ++i) {
                const float sc = __fmul_rn(d[i], ubyte_f<u & 3>(scw[i][u >> 2], 0x3Fu));
                const float mn = __fmul_rn(dmin[i], ubyte_f<u & 3>(mnw[i][u >> 2], 0x3Fu));
                a2[i] = make_float2(sc, sc);
                nb2[i] = make_float2(-mn, -mn);
            }
            // qs words 4t..4t+3 of the pair are read as one 16-byte line when
            // the chain first needs them (4-byte reads at the 144-byte row
            // stride would hit 8 banks from 32 lanes)
            uint4 qv[NR0];
            chain_acc<M, NR0, 8, 256>(acc, xc + 32 * u, [&](auto qc, int i, float2& w01, float2& w23) {
                constexpr int Q = decltype(qc)::value;
                if constexpr ((Q & 3) == 0) qv[i] = lds16(rows[i] + 16 + 32 * cq + 4 * Q);
                q4k_group<H>(word_of<Q & 3>(qv[i]), w01, w23);
                w01 = fma2(a2[i], w01, nb2[i]);
                w23 = fma2(a2[i], w23, nb2[i]);
            });
        });
    });
}

// Affine: values 4Q..4Q+3 of a staged row from their code word v (word Q
// for 8-bit codes, word Q/2 for 4-bit).  4-bit codes sit lowest-first, 8 per
// word: values 0..3 of a word at bits 0, 4, 8, 12 (exponents 2^23, 2^19,
// 2^15, 2^11), values 4..7 at bits 16 and (after >> 12) 8, 12, 16.  8-bit
// codes are the word's bytes.
template <int BITS, int Q>
__device__ __forceinline__ void affine_codes(uint32_t v, float2& w01, float2& w23) {
    if constexpr (BITS == 8) {
        const float2 bias = make_float2(-8388608.0f, -32768.0f);
        w01 = bytes01_u(v, 0xFFu, 0xFF00u, bias);
        w23 = bytes01_u(v >> 16, 0xFFu, 0xFF00u, bias);
    } else {
        if constexpr ((Q & 1) == 0) {
            w01 = add2(make_float2(fbits(lop_and_or(v, 0xFu, 0x4B000000u)), fbits(lop_and_or(v, 0xF0u, 0x49000000u))),
                       make_float2(-8388608.0f, -524288.0f));
            w23 = add2(make_float2(fbits(lop_and_or(v, 0xF00u, 0x47000000u)), fbits(lop_and_or(v, 0xF000u, 0x45000000u))),
                       make_float2(-32768.0f, -2048.0f));
        } else {
            const uint32_t sh = v >> 12;
            w01 = add2(make_float2(fbits(lop_and_or(v, 0xF0000u, 0x43000000u)), fbits(lop_and_or(sh, 0xF00u, 0x47000000u))),
                       make_float2(-128.0f, -32768.0f));
            w23 = add2(make_float2(fbits(lop_and_or(sh, 0xF000u, 0x45000000u)), fbits(lop_and_or(sh, 0xF0000u, 0x43000000u))),
                       make_float2(-2048.0f, -128.0f));
        }
    }
}

// Affine, 3, 5 or 6 bits: the four codes at bits 0, BITS, 2*BITS and 3*BITS
// of v (a window of the row's bit stream) as exact floats: each field goes
// in as mantissa bits under the exponent that puts its lowest bit at 2^0
// (2^23 for bit 0, 2^(23-BITS) for bit BITS), and the exponent's value is
// subtracted; the upper pair is read the same way from v >> 2*BITS.
template <int BITS>
__device__ __forceinline__ void affine_codes_n(uint32_t v, float2& w01, float2& w23) {
    constexpr uint32_t M = (1u << BITS) - 1u;
    constexpr uint32_t E1 = static_cast<uint32_t>(150 - BITS) << 23;
    const float2 bias = make_float2(-8388608.0f, -static_cast<float>(1u << (23 - BITS)));
    const uint32_t u = v >> (2 * BITS);
    w01 = add2(make_float2(fbits(lop_and_or(v, M, 0x4B000000u)), fbits(lop_and_or(v, M << BITS, E1))), bias);
    w23 = add2(make_float2(fbits(lop_and_or(u, M, 0x4B000000u)), fbits(lop_and_or(u, M << BITS, E1))), bias);
}

// Word W (0..7) of two 16-byte lines.
template <int W>
__device__ __forceinline__ uint32_t word8(const uint4& a, const uint4& b) {
    if constexpr (W < 4) return word_of<W>(a);
    else return word_of<W - 4>(b);
}

// Affine chunk: every weight is dequantized on its own, w = fl(fl(scale*q) +
// bias); scale*q (a binary16 times a code of at most 8 bits) is exact in
// binary32, so that is fma(scale, q, bias) bit for bit.  Then acc += w*x.
// Scales and biases come from global memory; rows past n and groups past k
// (a last chunk that ends inside the row) read none, and their zero scale
// and bias give weights of exactly zero.  The lane holds NR0 rows (warp row
// rl + LW*i); xl is its first input row.
template <int M, int NR0, int LW, int WT>
__device__ __forceinline__ void chunk_affine(const uint8_t* const (&rows)[NR0], const float* xl, int rl,
                                             const MvArgs& a, uint32_t b, uint32_t wrow0, uint32_t cc,
                                             float2 (&acc)[NR0][M]) {
    constexpr int BITS = affine_bits(WT), GS = affine_group(WT);
    constexpr int CV = Stage<WT>::kValues, NG = CV / GS;
    uint64_t base[NR0];
    bool live[NR0];
#pragma unroll
    for (int i = 0; i < NR0; ++i) {
        const uint32_t row = wrow0 + static_cast<uint32_t>(rl + LW * i);
        live[i] = row < a.n;
        base[i] = (static_cast<uint64_t>(b) * a.n + row) * a.ngroups + static_cast<uint64_t>(cc) * NG;
    }
    static_for<0, NG>([&](auto gc) {
        constexpr int g = decltype(gc)::value;
        float2 sc2[NR0], bi2[NR0];
#pragma unroll
        for (int i = 0; i < NR0; ++i) {
            const bool on = live[i] && cc * NG + g < a.ngroups;
            const float sc = on ? h2f(__ldg(a.scales + base[i] + g)) : 0.0f;
            const float bi = on ? h2f(__ldg(a.biases + base[i] + g)) : 0.0f;
            sc2[i] = make_float2(sc, sc);
            bi2[i] = make_float2(bi, bi);
        }
        if constexpr (BITS == 4 || BITS == 8) {
            // code words are read as 16-byte lines when the chain first needs
            // them (a group's codes are a whole number of lines)
            uint4 cv[NR0];
            chain_acc<M, NR0, GS / 4, CV>(acc, xl + GS * g, [&](auto qc, int i, float2& w01, float2& w23) {
                constexpr int Q = g * (GS / 4) + decltype(qc)::value;
                constexpr int WI = BITS == 8 ? Q : Q / 2;  // code word of values 4Q..4Q+3
                if constexpr ((WI & 3) == 0 && (BITS == 8 || (Q & 1) == 0)) cv[i] = lds16(rows[i] + 4 * WI);
                affine_codes<BITS, Q>(word_of<WI & 3>(cv[i]), w01, w23);
                w01 = fma2(sc2[i], w01, bi2[i]);
                w23 = fma2(sc2[i], w23, bi2[i]);
            });
        } else {
            // 3, 5 or 6 bits: 32 values (4*BITS bytes, from byte 4*BITS*SG of
            // the chunk) lie in at most two 16-byte lines, read when the
            // chain reaches them; quad QQ of the 32 takes the 4*BITS stream
            // bits from bit 4*BITS*QQ on, one word or a funnel shift of two
            uint4 la[NR0], lb[NR0];
            chain_acc<M, NR0, GS / 4, CV>(acc, xl + GS * g, [&](auto qc, int i, float2& w01, float2& w23) {
                constexpr int Q = g * (GS / 4) + decltype(qc)::value;  // quad of the chunk
                constexpr int SG = Q / 8, QQ = Q % 8;
                constexpr int L0 = (4 * BITS * SG) / 16, L1 = (4 * BITS * SG + 4 * BITS - 1) / 16;
                static_assert(L1 <= L0 + 1, "32 values span at most two lines");
                if constexpr (QQ == 0) {
                    la[i] = lds16(rows[i] + 16 * L0);
                    if constexpr (L1 > L0) lb[i] = lds16(rows[i] + 16 * L1);
                }
                constexpr int B = 32 * BITS * SG + 4 * BITS * QQ - 128 * L0;  // first bit, from line L0
                constexpr int WI = B / 32, S = B % 32;
                uint32_t v;
                if constexpr (S + 4 * BITS <= 32) v = word8<WI>(la[i], lb[i]) >> S;
                else v = __funnelshift_r(word8<WI>(la[i], lb[i]), word8<WI + 1>(la[i], lb[i]), S);
                affine_codes_n<BITS>(v, w01, w23);
                w01 = fma2(sc2[i], w01, bi2[i]);
                w23 = fma2(sc2[i], w23, bi2[i]);
            });
        }
    });
}

// Q6_K super-block staged at byte o of each row: 16 sub-blocks of 16
// values, u = 8h + 2t + gh, each its own chain scaled by d * sc[u].
template <int M, int NR0>
__device__ __forceinline__ void chunk_q6_k(const uint8_t* const (&rows)[NR0], const float* xc, int o,
                                           float2 (&acc)[NR0][M]) {
    uint32_t wd[NR0][53];
    float d[NR0];
#pragma unroll
    for (int i = 0; i < NR0; ++i) {
        q6_load(rows[i], o, wd[i]);
        d[i] = h2f(wd[i][52]);
    }
    static_for<0, 16>([&](auto uc) {
        constexpr int u = decltype(uc)::value;
        constexpr int h = u >> 3, t = (u >> 1) & 3, gh = u & 1;
        float a[NR0];
#pragma unroll
        for (int i = 0; i < NR0; ++i) a[i] = __fmul_rn(d[i], sbyte_f<u & 3>(wd[i][48 + (u >> 2)]));
        float2 c[NR0][M];
        chain<M, NR0, 4, 256>(c, xc + 128 * h + 32 * t + 16 * gh, [&](auto qc, int i, float2& w01, float2& w23) {
            q6k_group<h, t, 4 * gh + decltype(qc)::value>(wd[i], w01, w23);
        });
        apply_scale<M, NR0>(acc, c, a);
    });
}

// ---------------------------------------------------------------- staging

// Fallback staging (the TMA path needs 16-byte aligned rows), done by the
// producer warp: chunk cc of `nrows` weight rows, copied with 2-byte loads
// (W only needs 2-byte alignment) into the positions a TMA box uses.  The
// staged row's bytes outside the chunk read as zero, as a TMA box past the
// row end does.
template <int WT>
__device__ __forceinline__ void stage_w_plain(uint8_t* dst_rows, const uint8_t* wrow0, uint64_t row_bytes,
                                              int nrows, uint32_t cc, uint32_t k, int lane) {
    constexpr int BOX = Stage<WT>::kBox;
    uint32_t first, len;  // byte range of the chunk inside the row
    if constexpr (is_affine(WT)) {
        first = cc * Stage<WT>::kBytes;
        len = static_cast<uint32_t>(min(static_cast<uint64_t>(Stage<WT>::kBytes), row_bytes - first));
    } else if constexpr (WT == kF16 || WT == kBF16) {
        first = cc * 144u;
        len = 2u * min(72u, k - cc * 72u);
    } else if constexpr (WT == kF32) {
        first = cc * 144u;
        len = 4u * min(36u, k - cc * 36u);
    } else if constexpr (WT == kQ8_0) {
        first = cc * 136u;
        len = min(4u, k / 32u - cc * 4u) * 34u;
    } else if constexpr (WT == kQ5_0) {
        first = cc * 176u;
        len = min(8u, k / 32u - cc * 8u) * 22u;
    } else if constexpr (WT == kQ4_K) {
        first = cc * 144u;
        len = 144u;
    } else {
        first = cc * 210u;
        len = 210u;
    }
    const uint32_t so = static_cast<uint32_t>(Stage<WT>::sofs(cc));
    for (int r = 0; r < nrows; ++r) {
        const uint16_t* src = reinterpret_cast<const uint16_t*>(wrow0 + static_cast<uint64_t>(r) * row_bytes + first);
        uint16_t* dst = reinterpret_cast<uint16_t*>(dst_rows + r * BOX);
        for (uint32_t h = lane; h < static_cast<uint32_t>(BOX / 2); h += 32) {
            const uint32_t p = 2u * h;
            dst[h] = (p >= so && p < so + len) ? __ldg(src + ((p - so) >> 1)) : static_cast<uint16_t>(0);
        }
    }
}

// Fallback input staging by the producer warp: the [M][CV] slice of chunk
// cc, zero past k.
template <int M, int CV>
__device__ __forceinline__ void stage_x_plain(float* dst, const float* xb, uint32_t xrs, uint32_t cc, uint32_t k,
                                              int lane) {
    constexpr int Q = CV / 4;
    for (int idx = lane; idx < M * Q; idx += 32) {
        const int j = idx / Q, q = idx - (idx / Q) * Q;
        const uint32_t col = cc * CV + 4u * q;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (col < k) v = ldg4(xb + static_cast<uint64_t>(j) * xrs + col);
        *reinterpret_cast<float4*>(dst + j * CV + 4 * q) = v;
    }
}

// Plain input staging for runtime m (the tensor-core kernel, whose tile is
// wider than the launch's m): the [m][CV] slice of chunk cc, zero past k.
template <int CV>
__device__ __forceinline__ void stage_x_plain_m(float* dst, const float* xb, uint32_t xrs, uint32_t m, uint32_t cc,
                                                uint32_t k, int lane) {
    constexpr int Q = CV / 4;
    for (int idx = lane; idx < static_cast<int>(m) * Q; idx += 32) {
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

// A lane's share of its warp's work under lane layout (NR0, H): the lanes
// form H groups of LW = 32/H; lane l holds the R = NR0*H warp rows
// rl + LW*i (rl = l % LW) and the MH = ceil(M/H) input rows mb .. mb+MH-1,
// mb = min(g*MH, M - MH) for its group g.  With odd M the last group starts
// early and repeats input rows of the group before it; those slots are
// computed (identically) but stored by their owner only.
template <int M, int NR0, int H>
struct LaneMap {
    static constexpr int R = NR0 * H;
    static constexpr int MH = (M + H - 1) / H;
    static constexpr int LW = kLanes / H;
    __device__ __forceinline__ static int rl(int lane) { return lane % LW; }
    __device__ __forceinline__ static int grp(int lane) { return lane / LW; }
    __device__ __forceinline__ static int mb(int lane) { return min(grp(lane) * MH, M - MH); }
    // slot j of the lane is its group's own input row (not a repeat)
    __device__ __forceinline__ static bool owns(int lane, int j) { return mb(lane) + j >= grp(lane) * MH; }
};

// Decode + multiply one staged chunk for the lane's rows.
template <int WT, int M, int NR0, int H>
__device__ __forceinline__ void mv_chunk(const uint8_t* st, uint32_t wstage, int warp, int lane, uint32_t cc,
                                         float2 (&acc)[NR0 * H][(M + H - 1) / H], const MvArgs& a, uint32_t b,
                                         uint32_t wrow0) {
    using L = LaneMap<M, NR0, H>;
    constexpr int R = L::R, MH = L::MH, LW = L::LW;
    constexpr int BOX = Stage<WT>::kBox;
    constexpr int CV = Stage<WT>::kValues;
    constexpr int ROWS = kLanes * NR0;
    const int rl = L::rl(lane), mb = L::mb(lane);
    const uint8_t* rows[R];
#pragma unroll
    for (int i = 0; i < R; ++i) rows[i] = st + (warp * ROWS + rl + LW * i) * BOX;
    const float* xc = reinterpret_cast<const float*>(st + wstage);  // [M][CV]
    const float* xl = xc + mb * CV;                                  // the lane's first input row
    if constexpr (is_affine(WT)) {
        chunk_affine<MH, R, LW, WT>(rows, xl, rl, a, b, wrow0, cc, acc);
    } else if constexpr (WT == kF16) {
        chunk_f16<MH, R>(rows, xl, acc);
    } else if constexpr (WT == kBF16 || WT == kF32) {
        chunk_dense<MH, R, WT>(rows, xl, acc);
    } else if constexpr (WT == kQ8_0) {
        if (Stage<WT>::sofs(cc) == 0) chunk_blocks32<MH, R, BlkQ8, 4, 34, 0>(rows, xl, acc);
        else chunk_blocks32<MH, R, BlkQ8, 4, 34, 8>(rows, xl, acc);
    } else if constexpr (WT == kQ5_0) {
        chunk_blocks32<MH, R, BlkQ5, 8, 22, 0>(rows, xl, acc);
    } else if constexpr (WT == kQ4_K) {
        chunk_q4_k<MH, R>(rows, xl, acc);
    } else {
        static_assert(WT != kQ6_K || H == 1, "Q6_K keeps one lane group");
        chunk_q6_k<MH, R>(rows, xl, Stage<WT>::sofs(cc), acc);
    }
}

// End of a row block for one consumer warp, given the lane's range partials
// part[i][j] of output row wrow0 + rl + LW*i and input row mb + j: either the
// store (split 1) or the in-order sum of the cluster's ranges.  With split S
// every rank publishes its partials in shared memory, one cluster barrier
// makes them visible, and slot (i, j) of each lane is finished by rank
// (i*MH + j) mod S: it loads the S partials of that output (its own and the
// peers', through distributed shared memory), all loads issued before the
// first add, and adds them in rank order.  Slots for which owns(j) is false
// (an input row another lane group stores, or one past the launch's m) are
// neither finished nor stored; a warp that is no holder (its partials were
// already added into another warp's) only takes part in the barrier.  Every
// thread of every CTA of the cluster reaches the cluster barrier once per row
// block.
// parts holds two buffers (row-block parities) buf_stride floats apart.
template <int R, int MH, int LW, typename Owns>
__device__ __forceinline__ void finish_row_block(const float (&part)[R][MH], const MvArgs& a, uint32_t b,
                                                 uint32_t wrow0, bool wactive, int rl, int mb, int lane, int warp,
                                                 uint32_t s, uint32_t S, uint32_t t, float* parts,
                                                 uint32_t buf_stride, Owns&& owns, bool holder = true) {
    // the store, with the optional epilogue alpha * acc + beta * c (each output
    // element on its own, after the fixed reduction: row exactness is kept)
    auto store = [&](int i, int j, float v) {
        const uint32_t row = wrow0 + static_cast<uint32_t>(rl + LW * i);
        const uint64_t m = static_cast<uint64_t>(mb + j);
        if (row >= a.n) return;
        if (a.epi == 1) {
            v = __fmul_rn(a.alpha, v);
        } else if (a.epi == 2) {
            const float cv = a.c[static_cast<uint64_t>(b) * a.cbs + m * a.crs + row];
            v = __fmaf_rn(a.alpha, v, __fmul_rn(a.beta, cv));
        }
        a.y[static_cast<uint64_t>(b) * a.ybs + m * a.yrs + row] = v;
    };
    if (S == 1) {
        if (wactive && holder) {
#pragma unroll
            for (int i = 0; i < R; ++i)
#pragma unroll
                for (int j = 0; j < MH; ++j)
                    if (owns(j)) store(i, j, part[i][j]);
        }
        return;
    }
    float* buf = parts + (t & 1u) * buf_stride;
    if (holder) {
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
            for (int j = 0; j < MH; ++j) buf[((warp * R + i) * MH + j) * 32 + lane] = part[i][j];
    }
    cluster_sync();  // phase t: the ranges' partials of this row block are published
    if (wactive && holder) {
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
            for (int j = 0; j < MH; ++j) {
                if (static_cast<uint32_t>(i * MH + j) % S != s || !owns(j)) continue;
                const float* slot = buf + ((warp * R + i) * MH + j) * 32 + lane;
                float p[kMaxSplit];
#pragma unroll
                for (int r = 0; r < kMaxSplit; ++r)
                    if (static_cast<uint32_t>(r) < S) p[r] = static_cast<uint32_t>(r) == s ? part[i][j] : ld_peer(slot, r);
                float v = p[0];
#pragma unroll
                for (int r = 1; r < kMaxSplit; ++r)
                    if (static_cast<uint32_t>(r) < S) v = __fadd_rn(v, p[r]);
                store(i, j, v);
            }
    }
}

// The lanes-over-rows kernel's finish: a range's partial is acc.x + acc.y
// (NaN for every output when a wait ran out), then finish_row_block.
template <int M, int NR0, int H>
__device__ __forceinline__ void mv_finish(const float2 (&acc)[NR0 * H][(M + H - 1) / H], bool failed,
                                          const MvArgs& a, uint32_t b, uint32_t wrow0, bool wactive, int lane,
                                          int warp, uint32_t s, uint32_t S, uint32_t t, float* parts,
                                          uint32_t part_floats) {
    using L = LaneMap<M, NR0, H>;
    constexpr int R = L::R, MH = L::MH, LW = L::LW;
    float part[R][MH];
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int j = 0; j < MH; ++j)
            part[i][j] = failed ? __int_as_float(0x7FC00000) : __fadd_rn(acc[i][j].x, acc[i][j].y);
    finish_row_block<R, MH, LW>(part, a, b, wrow0, wactive, L::rl(lane), L::mb(lane), lane, warp, s, S, t, parts,
                                part_floats, [&](int j) { return L::owns(lane, j); });
}

// ---------------------------------------------------------------- the kernel

// Persistent kernel (at most 4 consumer warps per CTA: 128 weight rows with
// one row per lane, 256 with two).  A cluster of `split` CTAs walks the row blocks
// cid, cid + nclusters, ... (a row block is G row groups of ROWS = 32*NR0
// rows of one batch); CTA rank s of the cluster handles K range s of every
// row block.  A CTA has G consumer warps (one row group each) and one
// producer warp.  Each pipeline stage holds one box of the row block's rows
// (G*ROWS x BOX bytes) and one box of the matching inputs (M x CV floats).
// The producer fills a stage once all consumer warps released it (mbarrier
// `empty`, G arrivals) and runs on into the next row block; consumers wait
// for the bytes (mbarrier `full`) and release each stage as soon as they are
// done with it.  The producer fills stages with TMA copies (rows 16-byte
// aligned) or, as a fallback, with plain loads and stores by its 32 lanes,
// each of which then arrives on `full`; the consumers run the same code
// either way.  After a row block every rank leaves its partial sums in
// shared memory (double-buffered by row-block parity), one cluster barrier
// publishes them, and each output is finished by one rank, which adds the
// ranges' partials in range order through distributed shared memory and
// stores y (see mv_finish).  The producer takes part in that barrier
// split-phase (arrive after issuing a row block, wait one row block later),
// so it never stalls the stream.
template <int WT, int M, int NR0, int H>
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
    constexpr int R = LaneMap<M, NR0, H>::R, MH = LaneMap<M, NR0, H>::MH;
    const uint32_t part_floats = static_cast<uint32_t>(G * R * MH * 32);
    float* parts = reinterpret_cast<float*>(smem + D * stage_bytes);  // [2][G][R][MH][32] when S > 1
    uint64_t* full = reinterpret_cast<uint64_t*>(parts + (S > 1 ? 2 * part_floats : 0));
    uint64_t* empty = full + kMaxStages;
    const uint32_t c0 = static_cast<uint32_t>((static_cast<uint64_t>(s) * a.nchunk) / S);
    const uint32_t c1 = static_cast<uint32_t>((static_cast<uint64_t>(s + 1) * a.nchunk) / S);
    const int nck = static_cast<int>(c1 - c0);
    const uint32_t nblocks = a.cpb * a.batch;  // row blocks of the whole launch

    // row block -> (batch, first row in the batch)
    auto block_origin = [&](uint32_t rb, uint32_t& b, uint32_t& row0) {
        b = rb / a.cpb;
        row0 = (rb - b * a.cpb) * static_cast<uint32_t>(G * ROWS);
    };

    const uint32_t fb = smem_u32(full), eb = smem_u32(empty);
    if (threadIdx.x == 0) {
        for (int t = 0; t < D; ++t) {
            mbar_init(fb + 8 * t, a.aligned ? 1u : 32u);
            mbar_init(eb + 8 * t, static_cast<uint32_t>(G));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // Launched as a programmatic dependent (a.pdl): the first row block's
    // weights go to L2 before the wait for the previous kernel (a prefetch
    // only fills L2, which every later write also goes through, so it cannot
    // make a later load stale); everything that reads x or W into shared
    // memory, or writes y, comes after the wait.  Without such a launch the
    // wait returns at once.
    if (a.pdl && a.aligned && producer && lane == 0 && cid < nblocks) {
        uint32_t b, row0;
        block_origin(cid, b, row0);
        const int32_t grow = static_cast<int32_t>(static_cast<uint64_t>(b) * a.n + row0);
        const int npf = min(nck, static_cast<int>(kPrefetchBytes / wstage) + 1);
        for (int q = 0; q < npf; ++q)
            tma_prefetch_2d(&wmap, static_cast<int32_t>(Stage<WT>::gofs(c0 + static_cast<uint32_t>(q)) / 2), grow);
    }
    pdl_wait();
    __syncthreads();

    if (producer) {
        // the next kernel of the stream may start its prologue now (it waits
        // for this one to complete before it touches memory this one writes)
        pdl_launch_dependents();
        uint32_t i = 0;  // running chunk counter over all row blocks
        bool stop = false;
        uint32_t t = 0;
        // test hook: issue no copy for the first stage, so that its waits run out
        const bool skip_first = (a.test_flags & kTestSkipFirstStage) != 0u;
        for (uint32_t rb = cid; rb < nblocks; rb += ncl, ++t) {
            uint32_t b, row0;
            block_origin(rb, b, row0);
            const uint64_t grow0 = static_cast<uint64_t>(b) * a.n + row0;
            if (a.aligned) {
                if (lane == 0 && !stop) {
                    for (int q = 0; q < nck; ++q, ++i) {
                        const int st = static_cast<int>(i % D);
                        if (i >= static_cast<uint32_t>(D) &&
                            !mbar_wait(eb + 8 * st, static_cast<uint32_t>((i / D - 1) & 1), a.wait_ns)) {
                            report_timeout(a.status, kStatusWaitTimeout);
                            stop = true;
                            break;
                        }
                        if (skip_first && i == 0) continue;
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
            } else if (!stop) {
                const int nrows = static_cast<int>(min(static_cast<uint32_t>(G * ROWS), a.n - row0));
                const uint8_t* wrow_ptr = a.w + grow0 * a.row_bytes;
                const float* xb = a.x + static_cast<uint64_t>(b) * a.xbs;
                for (int q = 0; q < nck; ++q, ++i) {
                    const int st = static_cast<int>(i % D);
                    if (i >= static_cast<uint32_t>(D) &&
                        !__all_sync(0xFFFFFFFFu,
                                    mbar_wait(eb + 8 * st, static_cast<uint32_t>((i / D - 1) & 1), a.wait_ns))) {
                        if (lane == 0) report_timeout(a.status, kStatusWaitTimeout);
                        stop = true;
                        break;
                    }
                    const uint32_t cc = c0 + static_cast<uint32_t>(q);
                    uint8_t* sp = smem + st * stage_bytes;
                    stage_w_plain<WT>(sp, wrow_ptr, a.row_bytes, nrows, cc, a.k, lane);
                    stage_x_plain<M, CV>(reinterpret_cast<float*>(sp + wstage), xb, a.xrs, cc, a.k, lane);
                    mbar_arrive(fb + 8 * st);
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
        if (a.aligned && lane == 0) {
            const uint32_t issued = i;
            for (uint32_t r = issued > static_cast<uint32_t>(D) ? issued - D : 0u; r < issued; ++r)
                if (!(skip_first && r == 0))
                    (void)mbar_wait(fb + 8 * (r % D), static_cast<uint32_t>((r / D) & 1), a.wait_ns);
        }
        __syncwarp();
        if (S > 1) cluster_sync();
        return;
    }

    bool failed = false;
    int st = 0;          // stage of the current chunk
    uint32_t ph = 0;     // its full-barrier parity
    bool seen = false;   // a poll during the previous chunk found this stage full
    for (uint32_t rb = cid, t = 0; rb < nblocks; rb += ncl, ++t) {
        uint32_t b, row0;
        block_origin(rb, b, row0);
        const uint32_t wrow0 = row0 + static_cast<uint32_t>(warp * ROWS);
        const bool wactive = wrow0 < a.n;
        float2 acc[R][MH];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int j = 0; j < MH; ++j) acc[r][j] = make_float2(0.0f, 0.0f);
        for (int q = 0; q < nck; ++q) {
            const int st1 = st + 1 == D ? 0 : st + 1;
            const uint32_t ph1 = st + 1 == D ? ph ^ 1u : ph;
            if (!failed && !__all_sync(0xFFFFFFFFu, seen) &&
                !__all_sync(0xFFFFFFFFu, mbar_wait(fb + 8 * st, ph, a.wait_ns))) {
                failed = true;
                if (lane == 0) report_timeout(a.status, kStatusWaitTimeout);
            }
            // poll the next stage now; the answer is used a chunk later (the
            // blocking wait runs only where it found the stage not yet full)
            seen = !failed && mbar_test(fb + 8 * st1, ph1);
            if (failed) {  // keep walking so every barrier below is still reached
                st = st1;
                ph = ph1;
                continue;
            }
            if (wactive)
                mv_chunk<WT, M, NR0, H>(smem + st * stage_bytes, wstage, warp, lane, c0 + static_cast<uint32_t>(q),
                                        acc, a, b, wrow0);
            __syncwarp();
            if (lane == 0) mbar_arrive(eb + 8 * st);
            st = st1;
            ph = ph1;
        }
        mv_finish<M, NR0, H>(acc, failed, a, b, wrow0, wactive, lane, warp, s, S, t, parts, part_floats);
    }
    if (S > 1) cluster_sync();
}

}  // namespace dev
}  // namespace rem

// Kernel pointer of one instantiation.  Two rows per lane in one group
// (NR0 = 2) exist for every M, two lane groups (H = 2) from M = 2 up;
// neither for Q6_K, whose 53 staged words per row would not fit twice in
// registers (and whose decode, not the input loads, bounds it).  Both
// together (four rows per lane) exist for F16 and BF16 at M = 6 and 8, the
// only formats and sizes where they measured faster: every other format
// pays more for decoding each row twice than it saves on input loads, and an
// odd M wastes the repeated input row.
namespace rem {
template <int WT, int M, int NR0, int H>
inline const void* mv_kernel_ptr() {
    if constexpr ((NR0 == 2 && WT == kQ6_K) || (H == 2 && (M < 2 || WT == kQ6_K)) ||
                  (NR0 == 2 && H == 2 && ((M != 6 && M != 8) || (WT != kF16 && WT != kBF16)))) {
        return nullptr;
    } else {
        return reinterpret_cast<const void*>(&dev::rem_mv_kernel<WT, M, NR0, H>);
    }
}
}  // namespace rem

// Each translation unit instantiates a range of M values of one weight
// format and exposes them through a lookup function (by layout index:
// (NR0, H) = (1, 1), (2, 1), (1, 2), (2, 2)).
#define REM_LAYOUTS(WT, MM)                                                                      \
    {mv_kernel_ptr<WT, MM, 1, 1>(), mv_kernel_ptr<WT, MM, 2, 1>(), mv_kernel_ptr<WT, MM, 1, 2>(), \
     mv_kernel_ptr<WT, MM, 2, 2>()}
#define REM_INSTANTIATE(WT, NAME, M0, NM)                                                           \
    namespace rem {                                                                                 \
    const void* NAME(int m, int layout) {                                                           \
        static const void* const table[4][kNumLayouts] = {                                          \
            REM_LAYOUTS(WT, M0), REM_LAYOUTS(WT, (NM > 1 ? M0 + 1 : M0)),                           \
            REM_LAYOUTS(WT, (NM > 2 ? M0 + 2 : M0)), REM_LAYOUTS(WT, (NM > 3 ? M0 + 3 : M0))};      \
        if (m < M0 || m >= M0 + NM || layout < 0 || layout >= kNumLayouts) return nullptr;          \
        return table[m - M0][layout];                                                               \
    }                                                                                               \
    }
