// rem_tc.cuh -- the row-exact few-row mat-vec on the tensor cores (tcgen05),
// for the block-scaled weights Q8_0, Q5_0 and Q6_K.
//
// y[b, j, i] = sum_k W[b*n + i, k] * x[b, j, k]
// (mlx-native 0.18.0 src/ops/row_exact_matvec.rs, module doc).  For these
// formats every weight is w = a_u * (q - offset) with one scale a_u per block
// u (Q8_0 and Q5_0: d of a 32-value block; Q6_K: d * sc of a 16-value
// sub-block), so
//     y = sum_u a_u * sum_{k in u} (q_k - offset) * x_k.
// The integer codes q - offset are exact in bfloat16, and each input value is
// split into bfloat16 parts x = x_hi + x_lo + r with x_hi the upper half of
// its binary32 bits and x_lo = bf16_rn(x - x_hi), so |r| <= 2^-16 |x|.  One
// tcgen05.mma (M = 128 weight rows, K = 16 values, N = max(16, 2*MP)
// columns: the MP x_hi rows of the inputs, then the MP x_lo rows, then zero
// rows) gives, per block, the exact products (q - offset)*x_hi and
// (q - offset)*x_lo summed in binary32 in tensor memory; the consumer warps
// then form c = D_hi + D_lo and acc = fma(a_u, c, acc) per output, in block
// order.  The error against the exact sum is below 2^-15 * sum |w*x| plus the
// binary32 rounding of the sums, well inside the required 1e-4 * sum |w*x|.
//
// Row exactness.  Output (i, j) depends only on weight row i (lane i of the
// tile), the bits of input row j (columns j and MP + j of every B tile), and
// the fixed order of blocks and K ranges; the tensor core computes each
// output column on its own, so neither m nor the tile width MP a launch
// takes (1, 2, 4, 8, 16 or 32 rows, the inputs padded with zeros) nor
// anything else of the launch changes it.
//
// Work mapping.  A CTA owns a tile of 128 consecutive weight rows (TMEM lane
// 32*(w%4) + l holds row 32*(w%4) + l for lane l of consumer warp w) and one
// K range (`split` CTAs of a cluster share a tile, as in the lanes-over-rows
// kernel).  Warps: 8 consumers (two per lane quarter, each decoding two of a
// unit's four K-steps), one TMA producer, two MMA warps (the first owns the
// tensor memory).  A staged chunk's inputs become its B tile (shared memory,
// canonical K-major layout without swizzle), converted by the MMA warps for
// a few input rows and by the consumers for more.  Per unit of 64 values the
// consumers decode their rows' codes into bf16 pairs and store them to the
// unit's A slot in tensor memory; units are handed to the MMA warps in steps
// of one or two, each step slot with one A-ready and one D-ready mbarrier;
// an MMA warp issues the step's MMAs into the slots' D columns and commits;
// the consumers read D back and scale it when they take the slot again.
// Waits whose phase has long completed are polled a step ahead, so they cost
// nothing on the consumers' path.  The slots rotate, so decoding the next
// units overlaps the MMAs.
#pragma once
#include "rem_mv.cuh"

namespace rem {
namespace dev {

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Instruction descriptor of kind::f16: D f32, A and B bf16, both K-major,
// M = 128, N = n.
__host__ __device__ constexpr uint32_t tc_idesc(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) | (8u << 24);
}

// Shared-memory descriptor of a K-major tile without swizzle: core matrices of
// 8 rows x 16 bytes, the two core matrices of a K step 128 bytes apart (LBO),
// consecutive groups of 8 rows 256 bytes apart (SBO).
__device__ __forceinline__ uint64_t tc_bdesc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(128u >> 4) << 16) |
           (static_cast<uint64_t>(256u >> 4) << 32) | (1ull << 46);
}

// D[128 x N] (+)= A[128 x 16] (tensor memory) * B[16 x N] (shared memory).
__device__ __forceinline__ void tc_mma(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// The mbarrier receives one arrival when every MMA this thread issued so far
// has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// C consecutive 32-bit columns of the warp's 32 lanes into r[0..C-1] (C = 2,
// 4 or 8; the rest of r is left as it is).
template <int C, int N>
__device__ __forceinline__ void tmem_ld_narrow(uint32_t taddr, uint32_t* r) {
    static_assert(C <= N, "columns");
    if constexpr (C == 2) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(taddr)
                     : "memory");
    } else if constexpr (C == 4) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(taddr)
                     : "memory");
    } else {
        static_assert(C == 8, "2, 4 or 8 columns");
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                       "=r"(r[7])
                     : "r"(taddr)
                     : "memory");
    }
}

// N consecutive 32-bit columns of the warp's 32 lanes (N = 16, 32, 64).
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[N]) {
    if constexpr (N == 16) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
            "%15}, [%16];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
            : "r"(taddr)
            : "memory");
    } else {
        static_assert(N % 32 == 0, "16, 32 or 64 columns");
#pragma unroll
        for (int h = 0; h < N / 32; ++h) {
            uint32_t* q = r + 32 * h;
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
                "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
                : "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3]), "=r"(q[4]), "=r"(q[5]), "=r"(q[6]), "=r"(q[7]),
                  "=r"(q[8]), "=r"(q[9]), "=r"(q[10]), "=r"(q[11]), "=r"(q[12]), "=r"(q[13]), "=r"(q[14]),
                  "=r"(q[15]), "=r"(q[16]), "=r"(q[17]), "=r"(q[18]), "=r"(q[19]), "=r"(q[20]), "=r"(q[21]),
                  "=r"(q[22]), "=r"(q[23]), "=r"(q[24]), "=r"(q[25]), "=r"(q[26]), "=r"(q[27]), "=r"(q[28]),
                  "=r"(q[29]), "=r"(q[30]), "=r"(q[31])
                : "r"(taddr + 32u * h)
                : "memory");
        }
    }
}

// ---------------------------------------------------------------- bfloat16 pairs

// a - b on two bfloat16 lanes (exact here: the results are small integers).
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// bfloat16 pair (lo in bits 0..15, hi in bits 16..31), each rounded to nearest even.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
// Bytes 0 and 2 (pair 0) and bytes 1 and 3 (pair 1) of v, masked to `mask`
// (at most 7 bits), as bfloat16 pairs 128 + code, then minus `off2` (the
// pair 128 + offset): exact code - offset.
__device__ __forceinline__ void codes_bf16(uint32_t v, uint32_t mask, uint32_t off2, uint32_t& p0, uint32_t& p1) {
    p0 = bf16x2_sub(lop_and_or(v, mask, 0x43004300u), off2);
    p1 = bf16x2_sub(lop_and_or(v >> 8, mask, 0x43004300u), off2);
}

// N little-endian words starting at byte POS (even) of a 16-byte aligned
// staged row, read as whole 16-byte lines.
template <int POS, int N>
__device__ __forceinline__ void row_words(const uint8_t* row, uint32_t (&w)[N]) {
    constexpr int L0 = POS / 16;
    constexpr int LAST = (POS % 4 == 0) ? POS + 4 * N - 1 : POS + 4 * N + 1;  // last byte read
    constexpr int NL = LAST / 16 - L0 + 1;
    uint32_t P[4 * NL];
#pragma unroll
    for (int l = 0; l < NL; ++l) {
        const uint4 v = lds16(row + 16 * (L0 + l));
        P[4 * l] = v.x; P[4 * l + 1] = v.y; P[4 * l + 2] = v.z; P[4 * l + 3] = v.w;
    }
    constexpr int B0 = POS - 16 * L0;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        if constexpr (B0 % 4 == 0) w[i] = P[B0 / 4 + i];
        else w[i] = __byte_perm(P[B0 / 4 + i], P[B0 / 4 + i + 1], 0x5432);
    }
}

// ---------------------------------------------------------------- formats

// Int8 codes: bytes 0 and 2 (pair 0) and 1 and 3 (pair 1) of v as exact
// bfloat16 pairs.  The low 7 bits go in as 128 + (q & 127) and the sign bit
// as the subtrahend 128 or 256, so one subtraction gives q exactly.
__device__ __forceinline__ void s8_bf16(uint32_t v, uint32_t& p0, uint32_t& p1) {
    p0 = bf16x2_sub(lop_and_or(v, 0x007F007Fu, 0x43004300u), lop_and_or(v, 0x00800080u, 0x43004300u));
    const uint32_t w = v >> 8;
    p1 = bf16x2_sub(lop_and_or(w, 0x007F007Fu, 0x43004300u), lop_and_or(w, 0x00800080u, 0x43004300u));
}

// Per format.  A unit is one K-step of 16 values in each of the 4 MMA slots
// of a slot's A columns; warp group g of a lane quarter decodes slots 2g and
// 2g+1 (A columns 16g .. 16g+15) of every unit.
//   kUPC         units per staged chunk;
//   kPerm        order of the 16 values of a K-step in A's columns (0 =
//                natural, 1 = values 4i, 4i+2, 4i+1, 4i+3 for each group i of
//                4: the byte pairs a byte-parallel decode yields);
//   kRK          K-steps per accumulator region: 2 where a warp's two
//                K-steps are the halves of one 32-value scale block (their
//                MMAs accumulate into one region, read and scaled once), else 1;
//   kstep(u, s)  the K-step of the chunk in MMA slot s of unit u (the B tile
//                that MMA reads);
//   Regs         the words a consumer lane keeps from one load to the units
//                that decode them (kLoad(u): a load at unit u; kLastLoad: the
//                unit after whose load the staged weights are no longer read);
//   load<U>      16-byte shared loads at compile-time positions; a switch
//                picks the body for the runtime byte position (chunk offset o,
//                warp group g);
//   decode<U>    unit U's 32 codes of the lane's row (slots 2g, 2g+1) as 16
//                bfloat16 pairs, and the scales of its 2 / kRK regions.
// The mapping keeps the bytes a warp needs together, so each staged byte is
// read about once per lane.
template <int WT> struct TcFmt;

// Q8_0: a chunk is 4 blocks (d f16 | 32 int8), 128 values at byte o = 0 or 8
// of the staged window.  Warp group g decodes block 2u + g in unit u: its
// halves are K-steps 4u + 2g and 4u + 2g + 1, one scale block.
template <> struct TcFmt<kQ8_0> {
    static constexpr int kUPC = 2, kPerm = 1, kLastLoad = 1, kRK = 2;
    __host__ __device__ static constexpr int kstep(int u, int s) { return 4 * u + s; }
    __host__ __device__ static constexpr bool kLoad(int) { return true; }
    struct Regs {
        uint32_t q[8];  // the 32 codes
        float d;
    };
    // An empty asm that "changes" the words, so no decode from them is
    // computed ahead of the point it is called at (register lifetimes stay
    // one unit long).
    __device__ __forceinline__ static void pin(Regs& r) {
        asm volatile("" : "+r"(r.q[0]), "+r"(r.q[1]), "+r"(r.q[2]), "+r"(r.q[3]), "+r"(r.q[4]), "+r"(r.q[5]),
                     "+r"(r.q[6]), "+r"(r.q[7]), "+f"(r.d));
    }
    template <int P>
    __device__ __forceinline__ static void block(const uint8_t* row, Regs& r) {
        uint32_t dw[1];
        row_words<P, 1>(row, dw);
        row_words<P + 2, 8>(row, r.q);
        r.d = h2f(dw[0]);
    }
    template <int U>
    __device__ __forceinline__ static void load(const uint8_t* row, int o, int g, Regs& r) {
        switch ((o ? 4 : 0) + 2 * U + g) {
        case 0: block<0>(row, r); break;
        case 1: block<34>(row, r); break;
        case 2: block<68>(row, r); break;
        case 3: block<102>(row, r); break;
        case 4: block<8>(row, r); break;
        case 5: block<42>(row, r); break;
        case 6: block<76>(row, r); break;
        default: block<110>(row, r); break;
        }
    }
    template <int U>
    __device__ __forceinline__ static void decode(const Regs& r, uint32_t (&a)[16], float (&scale)[1]) {
#pragma unroll
        for (int i = 0; i < 8; ++i) s8_bf16(r.q[i], a[2 * i], a[2 * i + 1]);
        scale[0] = r.d;
    }
};

// Q5_0: a chunk is 8 blocks (d f16 | qh u32 | 16 nibble bytes), 256 values
// at byte 0 of the staged row.  Warp group g decodes block 2u + g in unit u:
// the low nibbles (values 0..15, K-step 4u + 2g) and the high ones (values
// 16..31, K-step 4u + 2g + 1) of the same bytes; bit 4 of value e is bit e
// of qh.
template <> struct TcFmt<kQ5_0> {
    static constexpr int kUPC = 4, kPerm = 1, kLastLoad = 3, kRK = 2;
    __host__ __device__ static constexpr int kstep(int u, int s) { return 4 * u + s; }
    __host__ __device__ static constexpr bool kLoad(int) { return true; }
    struct Regs {
        uint32_t qs[4], qh;
        float d;
    };
    __device__ __forceinline__ static void pin(Regs& r) {
        asm volatile("" : "+r"(r.qs[0]), "+r"(r.qs[1]), "+r"(r.qs[2]), "+r"(r.qs[3]), "+r"(r.qh), "+f"(r.d));
    }
    template <int P>
    __device__ __forceinline__ static void block(const uint8_t* row, Regs& r) {
        uint32_t q[6];
        row_words<P, 6>(row, q);  // d | qh | qs (22 bytes, plus 2)
        r.d = h2f(q[0]);
        r.qh = __byte_perm(q[0], q[1], 0x5432);
#pragma unroll
        for (int i = 0; i < 4; ++i) r.qs[i] = __byte_perm(q[1 + i], q[2 + i], 0x5432);
    }
    template <int U>
    __device__ __forceinline__ static void load(const uint8_t* row, int, int g, Regs& r) {
        switch (2 * U + g) {
        case 0: block<0>(row, r); break;
        case 1: block<22>(row, r); break;
        case 2: block<44>(row, r); break;
        case 3: block<66>(row, r); break;
        case 4: block<88>(row, r); break;
        case 5: block<110>(row, r); break;
        case 6: block<132>(row, r); break;
        default: block<154>(row, r); break;
        }
    }
    template <int U>
    __device__ __forceinline__ static void decode(const Regs& r, uint32_t (&a)[16], float (&scale)[1]) {
#pragma unroll
        for (int kh = 0; kh < 2; ++kh)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t nib = kh ? (r.qs[i] >> 4) : r.qs[i];
                const uint32_t v = lop_and_or(nib, 0x0F0F0F0Fu, spread4((r.qh >> (16 * kh + 4 * i)) & 0xFu));
                codes_bf16(v, 0x001F001Fu, 0x43104310u, a[8 * kh + 2 * i], a[8 * kh + 2 * i + 1]);
            }
        scale[0] = r.d;
    }
};

// Q6_K: a chunk is one super-block (ql u8[128] | qh u8[64] | sc int8[16] | d
// f16) at byte o (even, < 16) of the staged window; its K-steps are the 16
// sub-blocks in order, each one scale block.  Sub-block s = 8h + 2t + e holds
// values 128h + 32t + 16e + l (l < 16): low bits from ql[64h + 32(t&1) + 16e
// + l] (the low nibble for t < 2, the high one for t >= 2), high bits 2t,
// 2t+1 of qh[32h + 16e + l], scale d * sc[s].  Warp group g = h decodes
// sub-blocks 8h + 2u + e (e = 0, 1; MMA slots 2h + e) in unit u = t, so the
// 96 code bytes it loads once (four 16-byte runs of ql, two of qh) serve all
// four of its units.
template <> struct TcFmt<kQ6_K> {
    static constexpr int kUPC = 4, kPerm = 1, kLastLoad = 0, kRK = 1;
    __host__ __device__ static constexpr int kstep(int u, int s) { return 8 * (s >> 1) + 2 * u + (s & 1); }
    __host__ __device__ static constexpr bool kLoad(int u) { return u == 0; }
    struct Regs {
        uint32_t qa[2][4], qb[2][4], qh[2][4];  // per e: ql for t = 0, 2 and t = 1, 3; qh
        uint32_t sc0, sc1;                      // sc[8h .. 8h+3] and sc[8h+4 .. 8h+7]
        float d;
    };
    __device__ __forceinline__ static void pin(Regs& r) {
#pragma unroll
        for (int e = 0; e < 2; ++e)
            asm volatile("" : "+r"(r.qa[e][0]), "+r"(r.qa[e][1]), "+r"(r.qa[e][2]), "+r"(r.qa[e][3]), "+r"(r.qb[e][0]),
                         "+r"(r.qb[e][1]), "+r"(r.qb[e][2]), "+r"(r.qb[e][3]), "+r"(r.qh[e][0]), "+r"(r.qh[e][1]),
                         "+r"(r.qh[e][2]), "+r"(r.qh[e][3]));
        asm volatile("" : "+r"(r.sc0), "+r"(r.sc1), "+f"(r.d));
    }
    template <int O>
    __device__ __forceinline__ static void body(const uint8_t* row, int h, Regs& r) {
        uint32_t sc4[4], dw[1];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            row_words<O, 4>(row + 64 * h + 16 * e, r.qa[e]);
            row_words<O + 32, 4>(row + 64 * h + 16 * e, r.qb[e]);
            row_words<O + 128, 4>(row + 32 * h + 16 * e, r.qh[e]);
        }
        row_words<O + 192, 4>(row, sc4);
        row_words<O + 208, 1>(row, dw);
        r.sc0 = h ? sc4[2] : sc4[0];
        r.sc1 = h ? sc4[3] : sc4[1];
        r.d = h2f(dw[0]);
    }
    template <int U>
    __device__ __forceinline__ static void load(const uint8_t* row, int o, int g, Regs& r) {
        switch (o) {
        case 0: body<0>(row, g, r); break;
        case 2: body<2>(row, g, r); break;
        case 4: body<4>(row, g, r); break;
        case 6: body<6>(row, g, r); break;
        case 8: body<8>(row, g, r); break;
        case 10: body<10>(row, g, r); break;
        case 12: body<12>(row, g, r); break;
        default: body<14>(row, g, r); break;
        }
    }
    template <int U>
    __device__ __forceinline__ static void decode(const Regs& r, uint32_t (&a)[16], float (&scale)[2]) {
        const uint32_t scw = U < 2 ? r.sc0 : r.sc1;  // sc[8h + 2t + e] is byte 2(t%2) + e of it
        scale[0] = __fmul_rn(r.d, (U & 1) ? sbyte_f<2>(scw) : sbyte_f<0>(scw));
        scale[1] = __fmul_rn(r.d, (U & 1) ? sbyte_f<3>(scw) : sbyte_f<1>(scw));
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t ql = (U & 1) ? r.qb[e][i] : r.qa[e][i];
                // high bits 2t, 2t+1 of each qh byte -> bits 4, 5
                uint32_t v;
                if constexpr (U < 2) v = lop_sel(ql, r.qh[e][i] << (4 - 2 * U), 0x0F0F0F0Fu);
                else v = lop_sel(ql >> 4, r.qh[e][i] >> (2 * U - 4), 0x0F0F0F0Fu);
                codes_bf16(v, 0x003F003Fu, 0x43204320u, a[8 * e + 2 * i], a[8 * e + 2 * i + 1]);
            }
    }
};

// ---------------------------------------------------------------- the kernel

// Geometry shared by the kernel and the host (rem_internal.h mirrors it).
template <int WT, int MP>
struct TcGeom {
    using F = TcFmt<WT>;
    static constexpr int CV = Stage<WT>::kValues;           // values per chunk
    static constexpr int BOX = Stage<WT>::kBox;             // staged bytes per row
    static constexpr int NCOL = tc_ncol(MP);                // MMA N: x_hi rows, then x_lo rows (>= 16)
    static constexpr int KSTEPS = CV / 16;                  // K-steps per chunk
    static constexpr int BKSTEP = 32 * NCOL;                // B bytes per K-step (NCOL rows x 32 bytes)
    static constexpr int BCHUNK = KSTEPS * BKSTEP;          // B bytes per chunk
    static constexpr int KPW = tc_kpw(MP);                  // K-steps of a unit per consumer warp
    static constexpr int CW = tc_consumer_warps(MP);        // consumer warps
    static constexpr int GROUPS = CW / 4;                   // warps per lane quarter
    static constexpr int RK = tc_region_ksteps(WT, MP);     // K-steps per accumulator region
    static constexpr int RPW = KPW / RK;                    // regions per warp
    static constexpr int NS = tc_slots(WT, MP);             // A/D slots
    static constexpr int ACOLS = 32;                        // A columns per slot (4 K-steps)
    static constexpr int DCOLS = tc_regions(WT, MP) * NCOL; // D columns per slot
    static constexpr int TCOLS = tc_tmem_cols(WT, MP);      // tensor memory allocated
    static constexpr int THREADS = tc_threads(MP);
    // units a consumer warp takes per step (their slot waits, tensor-memory
    // stores and loads and hand-overs issued together): two where the ring
    // holds two steps and the accumulators of two units fit in registers
    static constexpr int BATCH = (NS >= 4 && RPW * NCOL <= 32) ? 2 : 1;
    static_assert(F::kUPC == tc_units_per_chunk(WT), "units per chunk");
    static_assert(F::kUPC % NS == 0, "units per chunk must be a multiple of the slots");
    static_assert(KPW == 2 && RK == F::kRK && RPW * RK == KPW, "two K-steps per warp and unit, kRK per region");
    static_assert(NS * (ACOLS + DCOLS) <= TCOLS, "slots exceed the tensor memory");
    static_assert(F::kUPC % BATCH == 0 && NS % BATCH == 0, "steps of whole units");
    // step slots: the BATCH consecutive slots of a step share one A-ready and
    // one D-ready barrier, and one MMA warp issues the step's MMAs
    static constexpr int NSS = NS / BATCH;
    static constexpr int SPC = F::kUPC / BATCH;  // steps per chunk
    static_assert(SPC % NSS == 0, "steps per chunk must be a multiple of the step slots");
};

// Conversion of one chunk's inputs ([m][CV] binary32 at xs) into the B tiles
// at bt by the consumer warps: K-step s, logical value v (A column order) of
// input row j -> x_hi at tile row j, x_lo at tile row MP + j.  Work item r of
// input row j = one 16-byte row of a core matrix (logical values 8r .. 8r+7 of
// K-step r/2, half r%2), read as 32 contiguous bytes of the staged row.  Input
// rows lie a multiple of 128 bytes apart, so the bank of a read depends on r
// alone and the bank of a tile store on j alone: lane i of each quarter warp
// takes row 8*pass + i and item (b + i) mod 32, b = 4*warp + quarter, and
// lanes 4..7 read their second 16 bytes first, so the eight 16-byte reads and
// the eight stores of a quarter warp each fall in eight different banks.
// Rows m..MP-1 stay zero.
template <int WT, int MP>
__device__ __forceinline__ void tc_convert_x(const float* xs, uint8_t* bt, uint32_t m, int tid) {
    using G = TcGeom<WT, MP>;
    constexpr int PER = 2 * G::KSTEPS;                      // items per input row (32 or 16)
    static_assert(G::CW == 8 && PER <= 32, "8 consumer warps x 4 quarters cover the 32 item slots of a row");
    const int lane = tid & 31, i = lane & 7;
    const int r = ((tid >> 5) * 4 + (lane >> 3) + i) & 31;  // the same for every pass
    const int sw = i >> 2;                                  // second half first
    if (r >= PER) return;
    const int s = r >> 1, kh = r & 1;
    uint8_t* bs = bt + s * G::BKSTEP + kh * 128;
    for (int j = i; j < static_cast<int>(m); j += 8) {
        const float* src = xs + j * G::CV + 8 * r;
        const float4 f0 = ldx4(src + 4 * sw), f1 = ldx4(src + 4 * (sw ^ 1));
        const float4 u = sw ? f1 : f0, v = sw ? f0 : f1;
        float e[8];
        if constexpr (TcFmt<WT>::kPerm == 1) {
            e[0] = u.x; e[1] = u.z; e[2] = u.y; e[3] = u.w; e[4] = v.x; e[5] = v.z; e[6] = v.y; e[7] = v.w;
        } else {
            e[0] = u.x; e[1] = u.y; e[2] = u.z; e[3] = u.w; e[4] = v.x; e[5] = v.y; e[6] = v.z; e[7] = v.w;
        }
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const uint32_t b0 = __float_as_uint(e[2 * p]), b1 = __float_as_uint(e[2 * p + 1]);
            hi[p] = __byte_perm(b0, b1, 0x7632);     // upper halves: x_hi of both values
            // x_lo = bf16_rn(x - x_hi); zero where x is not finite (x_hi keeps inf / NaN)
            const float r0 = (b0 & 0x7F800000u) == 0x7F800000u ? 0.0f : __fsub_rn(e[2 * p], __uint_as_float(b0 & 0xFFFF0000u));
            const float r1 = (b1 & 0x7F800000u) == 0x7F800000u ? 0.0f : __fsub_rn(e[2 * p + 1], __uint_as_float(b1 & 0xFFFF0000u));
            lo[p] = bf16x2_rn(r0, r1);
        }
        // tile rows: x_hi at j, x_lo at MP + j
        const int rl = MP + j;
        *reinterpret_cast<uint4*>(bs + (j >> 3) * 256 + (j & 7) * 16) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(bs + (rl >> 3) * 256 + (rl & 7) * 16) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

// One MMA warp's share of a chunk's inputs ([m][CV] binary32 at xs) in the B
// tiles at bt: the K-steps of the units that warp issues (its step slots),
// so no other warp's MMAs read what it writes.  K-step s, logical value v (A
// column order) of input row j -> x_hi at tile row j, x_lo at tile row MP +
// j.  Work item = one 16-byte row of a core matrix (8 logical values of one
// input row); rows m..MP-1 stay zero.
template <int WT, int MP>
__device__ __forceinline__ void tc_convert_x_part(const float* xs, uint8_t* bt, uint32_t m, int lane, int par) {
    using G = TcGeom<WT, MP>;
    using F = TcFmt<WT>;
    constexpr int NU = F::kUPC / 2;                         // units of one MMA warp per chunk
    constexpr int PER = 8 * NU;                             // items per input row: 4 K-steps x 2 halves per unit
    static_assert((PER & (PER - 1)) == 0, "items per row a power of two");
    for (int it = lane; it < static_cast<int>(m) * PER; it += kLanes) {
        const int j = it / PER, e = it % PER;
        const int ui = e >> 3, k4 = (e >> 1) & 3, kh = e & 1;
        // the warp's steps are those of parity par (the step slots alternate)
        const int u = (2 * (ui / G::BATCH) + par) * G::BATCH + ui % G::BATCH;
        const int s = F::kstep(u, k4);
        const float* src = xs + j * G::CV + 16 * s + 8 * kh;
        const float4 a4 = ldx4(src), b4 = ldx4(src + 4);
        float x[8];
        if constexpr (F::kPerm == 1) {
            x[0] = a4.x; x[1] = a4.z; x[2] = a4.y; x[3] = a4.w; x[4] = b4.x; x[5] = b4.z; x[6] = b4.y; x[7] = b4.w;
        } else {
            x[0] = a4.x; x[1] = a4.y; x[2] = a4.z; x[3] = a4.w; x[4] = b4.x; x[5] = b4.y; x[6] = b4.z; x[7] = b4.w;
        }
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const uint32_t b0 = __float_as_uint(x[2 * p]), b1 = __float_as_uint(x[2 * p + 1]);
            hi[p] = __byte_perm(b0, b1, 0x7632);     // upper halves: x_hi of both values
            // x_lo = bf16_rn(x - x_hi); zero where x is not finite (x_hi keeps inf / NaN)
            const float r0 = (b0 & 0x7F800000u) == 0x7F800000u ? 0.0f : __fsub_rn(x[2 * p], __uint_as_float(b0 & 0xFFFF0000u));
            const float r1 = (b1 & 0x7F800000u) == 0x7F800000u ? 0.0f : __fsub_rn(x[2 * p + 1], __uint_as_float(b1 & 0xFFFF0000u));
            lo[p] = bf16x2_rn(r0, r1);
        }
        // tile rows: x_hi at j, x_lo at MP + j
        uint8_t* bs = bt + s * G::BKSTEP + kh * 128;
        const int rl = MP + j;
        *reinterpret_cast<uint4*>(bs + (j >> 3) * 256 + (j & 7) * 16) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(bs + (rl >> 3) * 256 + (rl & 7) * 16) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

// 8*KPW columns of the warp's 32 lanes.
template <int KPW>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[8 * KPW]) {
    if constexpr (KPW == 1) {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                     "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                     : "memory");
    } else {
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
            "%14, %15, %16};" ::"r"(taddr),
            "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
            "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
            : "memory");
    }
}

// The RPW accumulator regions of a warp, their D columns loaded into d
// (region b at columns b*N on: x_hi of input rows 0..MP-1, then x_lo): c =
// D_hi + D_lo for each of the tile's MP input rows (rows past m hold zeros
// and are never stored) and acc = fma(scale_b, c, acc), region by region.
// Columns go in pairs through the f32x2 add and fma, which round each lane
// as the binary32 ops do; each column is computed on its own, so the tile
// width changes no bit of an output.
template <int MP, int RPW>
__device__ __forceinline__ void tc_scale(const uint32_t (&d)[RPW * tc_ncol(MP)], const float (&sc)[RPW],
                                         float (&acc)[MP]) {
    constexpr int NC = tc_ncol(MP);
#pragma unroll
    for (int b = 0; b < RPW; ++b) {
        const float2 s2 = make_float2(sc[b], sc[b]);
#pragma unroll
        for (int j = 0; j + 1 < MP; j += 2) {
            const float2 c = add2(make_float2(__uint_as_float(d[b * NC + j]), __uint_as_float(d[b * NC + j + 1])),
                                  make_float2(__uint_as_float(d[b * NC + MP + j]),
                                              __uint_as_float(d[b * NC + MP + j + 1])));
            const float2 r = fma2(s2, c, make_float2(acc[j], acc[j + 1]));
            acc[j] = r.x;
            acc[j + 1] = r.y;
        }
        if constexpr (MP & 1)
            acc[MP - 1] = __fmaf_rn(sc[b], __fadd_rn(__uint_as_float(d[b * NC + MP - 1]),
                                                     __uint_as_float(d[b * NC + 2 * MP - 1])),
                                    acc[MP - 1]);
    }
}

// Persistent kernel: clusters of `split` CTAs walk the 128-row tiles; CTA
// rank s of a cluster handles K range s of every tile.  Warps 0..CW-1 are
// consumers: warp w holds rows 32(w%4) .. 32(w%4)+31 of the tile (its TMEM
// lane quarter) and, as warp group g = w/4, the K-steps kstep(u, 2g) and
// kstep(u, 2g+1) of every unit u with their accumulator regions.  Warp CW is
// the producer (TMA or plain staging of weights and inputs); warps CW+1 and
// CW+2 issue the MMAs of the even and the odd step slots (a step is the
// one or two units the consumers hand over together), and warp CW+1 owns the
// tensor memory.  The warps of one lane quarter accumulate separately; at the
// end of a tile their partials are added in warp-group order.
template <int WT, int MP, bool CM>
__global__ void __launch_bounds__(TcGeom<WT, MP>::THREADS, 1)
rem_tc_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap, const MvArgs a) {
    using G = TcGeom<WT, MP>;
    using F = TcFmt<WT>;
    constexpr int NS = G::NS, UPC = F::kUPC, KPW = G::KPW, RK = G::RK, RPW = G::RPW;
    constexpr int CV = G::CV, BOX = G::BOX, ROWS = 128;
    constexpr int CW = G::CW, PRODUCER = CW, ISSUER = CW + 1, ISSUER2 = CW + 2;
    constexpr int NSS = G::NSS, SPC = G::SPC, BATCH = G::BATCH;
    // who converts a chunk's inputs into its B tile (CM, chosen by the host
    // from the number of input rows, tc_conv_mma): the two MMA warps, each
    // the K-steps of its own units between its steps, off the consumers'
    // path; or, for more rows, the consumer warps, where the work spreads
    // over all four SM sub-partitions

    static_assert(NSS % 2 == 0, "the two MMA warps take alternate step slots");
    constexpr uint32_t XPAD = (MP * CV * 4 + 127u) & ~127u;
    constexpr uint32_t WSTAGE = ROWS * BOX;
    constexpr uint32_t STAGE = WSTAGE + XPAD;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t S = a.split;
    const int D = static_cast<int>(a.stages);
    const uint32_t m = a.m;
    const uint32_t s = S > 1 ? cluster_rank() : 0u;
    const uint32_t cid = blockIdx.x / S;
    const uint32_t ncl = gridDim.x / S;
    uint8_t* btiles = smem + D * STAGE;                                    // [2][BCHUNK]
    // [2][GROUPS-1][4][MP][32] by row-block parity: the partials of warp
    // groups 1.. of each lane quarter; with split > 1 the cross-range partials
    // of a row block reuse its buffer's group 1 slots (a group 0 warp reads
    // every slot of its quarter before it writes that one, and the buffer of
    // the same parity is written again only after the next row block's
    // cluster barrier, which every reader of the partials has passed)
    float* pairs = reinterpret_cast<float*>(btiles + 2 * G::BCHUNK);
    constexpr uint32_t part_floats = 4u * MP * 32u;
    constexpr uint32_t pair_floats = (G::GROUPS - 1) * part_floats;
    float* parts = pairs;
    uint64_t* full = reinterpret_cast<uint64_t*>(pairs + 2 * pair_floats);
    uint64_t* empty = full + kMaxStages;
    uint64_t* afull = empty + kMaxStages;
    uint64_t* dfull = afull + 4;
    uint64_t* drain = dfull + 4;   // [2], one per MMA warp
    // [2][2]: MMA warp p's MMAs of the chunks of parity b have completed (the
    // readers of B tile buffer b, for that warp's K-steps)
    uint64_t* bfree = drain + 2;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bfree + 4);
    const uint32_t c0 = static_cast<uint32_t>((static_cast<uint64_t>(s) * a.nchunk) / S);
    const uint32_t c1 = static_cast<uint32_t>((static_cast<uint64_t>(s + 1) * a.nchunk) / S);
    const int nck = static_cast<int>(c1 - c0);
    const uint32_t nblocks = a.cpb * a.batch;

    auto block_origin = [&](uint32_t rb, uint32_t& b, uint32_t& row0) {
        b = rb / a.cpb;
        row0 = (rb - b * a.cpb) * static_cast<uint32_t>(ROWS);
    };

    const uint32_t fb = smem_u32(full), eb = smem_u32(empty), ab = smem_u32(afull), db = smem_u32(dfull);
    if (threadIdx.x == 0) {
        for (int t = 0; t < D; ++t) {
            mbar_init(fb + 8 * t, a.aligned ? 1u : 32u);
            mbar_init(eb + 8 * t, static_cast<uint32_t>(CW + 2));  // consumers and the two MMA warps
        }
        for (int t = 0; t < NSS; ++t) {
            mbar_init(ab + 8 * t, static_cast<uint32_t>(CW));
            mbar_init(db + 8 * t, 1u);
        }
        mbar_init(smem_u32(drain), 1u);
        mbar_init(smem_u32(drain + 1), 1u);
        for (int t = 0; t < 4; ++t) mbar_init(smem_u32(bfree + t), 1u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // the B tiles' rows m..MP-1 stay zero for the whole launch
    for (int i = threadIdx.x; i < 2 * G::BCHUNK / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(btiles)[i] = make_uint4(0u, 0u, 0u, 0u);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (a.pdl && a.aligned && warp == PRODUCER && lane == 0 && cid < nblocks) {
        uint32_t b, row0;
        block_origin(cid, b, row0);
        const int32_t grow = static_cast<int32_t>(static_cast<uint64_t>(b) * a.n + row0);
        const int npf = min(nck, static_cast<int>(kPrefetchBytes / WSTAGE) + 1);
        for (int q = 0; q < npf; ++q)
            tma_prefetch_2d(&wmap, static_cast<int32_t>(Stage<WT>::gofs(c0 + static_cast<uint32_t>(q)) / 2), grow);
    }
    pdl_wait();
    // tensor memory, once the previous kernel of the stream (which may have
    // held some) has completed
    if (warp == ISSUER) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "n"(G::TCOLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the same value in every lane, and known to the compiler to be so
    const uint32_t tmem = __shfl_sync(0xFFFFFFFFu, *tslot, 0);

    if (warp == PRODUCER) {
        // ------------------------------------------------ producer
        pdl_launch_dependents();
        uint32_t i = 0;
        bool stop = false;
        uint32_t t = 0;
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
                        uint8_t* sp = smem + st * STAGE;
                        mbar_expect_tx(fb + 8 * st, WSTAGE + m * CV * 4u);
                        tma_load_2d(smem_u32(sp), &wmap, static_cast<int32_t>(Stage<WT>::gofs(cc) / 2),
                                    static_cast<int32_t>(grow0), fb + 8 * st);
                        tma_load_3d(smem_u32(sp + WSTAGE), &xmap, static_cast<int32_t>(cc * CV),
                                    a.x_bm ? static_cast<int32_t>(b) : 0, a.x_bm ? 0 : static_cast<int32_t>(b),
                                    fb + 8 * st);
                    }
                }
            } else if (!stop) {
                const int nrows = static_cast<int>(min(static_cast<uint32_t>(ROWS), a.n - row0));
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
                    uint8_t* sp = smem + st * STAGE;
                    stage_w_plain<WT>(sp, wrow_ptr, a.row_bytes, nrows, cc, a.k, lane);
                    stage_x_plain_m<CV>(reinterpret_cast<float*>(sp + WSTAGE), xb, a.xrs, m, cc, a.k, lane);
                    mbar_arrive(fb + 8 * st);
                }
            }
            __syncwarp();
            if (S > 1) {
                if (t > 0) cluster_wait();
                cluster_arrive();
            }
        }
        if (S > 1 && t > 0) cluster_wait();
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

    if (warp == ISSUER || warp == ISSUER2) {
        // ------------------------------------------------ MMA issuers
        // Two warps issue the MMAs, the first for the even step slots, the
        // second for the odd ones: a commit and the wait on it before a slot
        // is reused hold up only the steps of that warp, so the other warp's
        // MMAs keep the tensor pipe busy meanwhile.  Each warp walks all the
        // steps, so every operand is warp-uniform (the descriptors are a base
        // plus compile-time steps); its lane 0 issues.
        const int par = warp - ISSUER;
        bool failed = false;
        bool issued_any = false;
        uint32_t gc = 0;  // chunks over all tiles
        uint32_t t = 0;
        constexpr uint32_t idesc = tc_idesc(G::NCOL);
        const uint64_t bdesc0 = tc_bdesc(__shfl_sync(0xFFFFFFFFu, smem_u32(btiles), 0));
        int st = 0;       // stage of the current chunk
        uint32_t ph = 0;  // its full-barrier parity
        for (uint32_t rb = cid; rb < nblocks; rb += ncl, ++t) {
            for (int q = 0; q < nck && !failed; ++q, ++gc) {
                const uint64_t bchunk = bdesc0 + static_cast<uint64_t>(((gc & 1u) * G::BCHUNK) >> 4);
                // where the MMA warps convert: this warp's K-steps of the
                // chunk's inputs -> B tile buffer gc & 1, once the chunk is
                // staged and this warp's MMAs of chunk gc - 2 (the buffer's
                // last readers of those K-steps) have completed
                const uint32_t bf = smem_u32(bfree + 2 * par + static_cast<int>(gc & 1u));
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(fb + 8 * st, ph, a.wait_ns)) ||
                    (CM && gc >= 2u &&
                     !__all_sync(0xFFFFFFFFu, mbar_wait(bf, ((gc >> 1) - 1u) & 1u, a.wait_ns)))) {
                    if (lane == 0) report_timeout(a.status, kStatusWaitTimeout);
                    failed = true;
                    break;
                }
                if constexpr (CM) {
                    tc_convert_x_part<WT, MP>(reinterpret_cast<const float*>(smem + st * STAGE + WSTAGE),
                                              btiles + (gc & 1u) * G::BCHUNK, m, lane, par);
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(eb + 8 * st);  // this warp has read the staged inputs
                if (++st == D) {
                    st = 0;
                    ph ^= 1u;
                }
                static_for<0, SPC>([&](auto p_) {
                    constexpr int P = decltype(p_)::value, SS = P % NSS;
                    if (SS % 2 != par || failed) return;
                    const uint32_t use = gc * (SPC / NSS) + static_cast<uint32_t>(P / NSS);
                    if (!__all_sync(0xFFFFFFFFu, mbar_wait(ab + 8 * SS, use & 1u, a.wait_ns))) {
                        if (lane == 0) report_timeout(a.status, kStatusWaitTimeout);
                        failed = true;
                        return;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        static_for<0, BATCH>([&](auto b_) {
                            constexpr int U = P * BATCH + decltype(b_)::value, SL = U % NS;
                            const uint32_t ac = tmem + static_cast<uint32_t>(SL * G::ACOLS);
                            const uint32_t dc = tmem + static_cast<uint32_t>(NS * G::ACOLS + SL * G::DCOLS);
#pragma unroll
                            for (int k4 = 0; k4 < 4; ++k4)
                                tc_mma(dc + static_cast<uint32_t>((k4 / RK) * G::NCOL), ac + 8u * k4,
                                       bchunk + static_cast<uint64_t>((F::kstep(U, k4) * G::BKSTEP) >> 4), idesc,
                                       (k4 % RK) != 0);
                        });
                        tc_commit(db + 8 * SS);
                    }
                    __syncwarp();
                    issued_any = true;
                });
                if (!failed && lane == 0) tc_commit(bf);
                __syncwarp();
            }
            if (S > 1) {
                if (t > 0) cluster_wait();
                cluster_arrive();
            }
        }
        if (S > 1 && t > 0) cluster_wait();
        if (S > 1) cluster_sync();
        // every MMA this warp issued has completed before the memory goes back
        if (lane == 0 && issued_any) {
            tc_commit(smem_u32(drain + par));
            if (!mbar_wait(smem_u32(drain + par), 0u, a.wait_ns)) report_timeout(a.status, kStatusWaitTimeout);
        }
        __syncwarp();
        asm volatile("bar.sync 1, %0;" ::"n"((CW + 2) * 32) : "memory");
        if (par == 0) {
            tc_fence_after();
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(G::TCOLS) : "memory");
        }
        return;
    }

    // ---------------------------------------------------- consumers
    const int quarter = warp & 3, grp = warp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;  // this warp's TMEM lanes
    // the words of unit b of a step come from Regs R[b] where every unit loads
    // its own, else all from R[0] (loaded once per chunk)
    constexpr bool kPerUnit = F::kLoad(1);
    bool failed = false;
    int st = 0;       // stage of the current chunk
    uint32_t ph = 0;  // its full-barrier parity
    uint32_t gc = 0;  // chunks over all tiles
    // wait for stage `sq` (unless an earlier poll, `seen`, found it full),
    // convert its inputs into B tile buffer `bsel` where the consumers do
    // that, and load unit 0's words of chunk q of the K range into r
    auto open_chunk = [&](int sq, uint32_t phase, int q, uint32_t bsel, typename F::Regs& r, bool seen = false) {
        if (!failed && !__all_sync(0xFFFFFFFFu, seen) &&
            !__all_sync(0xFFFFFFFFu, mbar_wait(fb + 8 * sq, phase, a.wait_ns))) {
            failed = true;
            if (lane == 0) report_timeout(a.status, kStatusWaitTimeout);
        }
        if (failed) return;
        const uint8_t* sp = smem + sq * STAGE;
        if constexpr (!CM) {
            tc_convert_x<WT, MP>(reinterpret_cast<const float*>(sp + WSTAGE), btiles + bsel * G::BCHUNK, m,
                                 static_cast<int>(threadIdx.x));
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        F::template load<0>(sp + (quarter * 32 + lane) * BOX, Stage<WT>::sofs(c0 + static_cast<uint32_t>(q)), grp,
                            r);
    };
    for (uint32_t rb = cid, t = 0; rb < nblocks; rb += ncl, ++t) {
        uint32_t b, row0;
        block_origin(rb, b, row0);
        const uint32_t wrow0 = row0 + static_cast<uint32_t>(quarter * 32);
        float acc[MP];
#pragma unroll
        for (int j = 0; j < MP; ++j) acc[j] = 0.0f;
        float psc[NS][RPW];  // region scales of the units in flight, by slot
#pragma unroll
        for (int j = 0; j < NS; ++j)
#pragma unroll
            for (int b = 0; b < RPW; ++b) psc[j][b] = 0.0f;
        // the step slot's MMAs (use number `use`) have completed: its D is
        // ready, its A is free
        auto wait_d = [&](int ss, uint32_t use) {
            if (failed) return;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(db + 8 * ss, use & 1u, a.wait_ns))) {
                failed = true;
                if (lane == 0) report_timeout(a.status, kStatusWaitTimeout);
                return;
            }
            tc_fence_after();
        };
        // the warp's RPW regions of slot sl: regions KPW*grp/RK on, contiguous
        // (the 1- and 2-row tiles read only their 2*MP used columns of each
        // region -- tc_scale reads no other; from 4 rows one wide load per
        // unit measured faster)
        auto load_d = [&](int sl, uint32_t (&d)[RPW * G::NCOL]) {
            const uint32_t ta = tmem + lane_base + static_cast<uint32_t>(NS * G::ACOLS + sl * G::DCOLS +
                                                                         (KPW * grp / RK) * G::NCOL);
            if constexpr (MP <= 2) {
#pragma unroll
                for (int r = 0; r < RPW; ++r)
                    tmem_ld_narrow<2 * MP, G::NCOL>(ta + static_cast<uint32_t>(r * G::NCOL), d + r * G::NCOL);
            } else {
                tmem_ld<RPW * G::NCOL>(ta, d);
            }
        };
        typename F::Regs R[kPerUnit ? BATCH : 1];
        // polls issued a step ahead: the next step's slot barrier (dseen) and,
        // from the chunk's first step, the next chunk's stage (fseen); the
        // blocking wait runs only where a poll found the phase incomplete
        bool dseen = false, fseen = false;
        // 1- and 2-row tiles of the formats that load a chunk's words once
        // (Q6_K): when the poll found the next step's slots complete, their
        // accumulators are read right away into dn (a few registers there),
        // so the read-back latency passes during the next step's decode;
        // dn_ok says it was done.  (Q8_0 and Q5_0, which load per unit,
        // measured slower with it.)
        constexpr bool kEarlyD = MP <= 2 && !kPerUnit;
        uint32_t dn[kEarlyD ? BATCH : 1][RPW * G::NCOL];
        bool dn_ok = false;
        // the first chunk of the tile; each later one is opened at the end of
        // the last step of the one before
        if (nck > 0) open_chunk(st, ph, 0, gc & 1u, R[0]);
        for (int q = 0; q < nck; ++q, ++gc) {
            if (failed) break;
            const uint8_t* row = smem + st * STAGE + (quarter * 32 + lane) * BOX;
            const int o = Stage<WT>::sofs(c0 + static_cast<uint32_t>(q));
            const bool more = q + 1 < nck;
            const int st1 = st + 1 == D ? 0 : st + 1;
            const uint32_t ph1 = st + 1 == D ? ph ^ 1u : ph;
            static_for<0, SPC>([&](auto p_) {
                constexpr int P = decltype(p_)::value, SS = P % NSS, U0 = BATCH * P;
                constexpr bool kLast = U0 + BATCH == UPC;
                if (failed) return;
                static_for<0, BATCH>([&](auto b_) {
                    constexpr int U = U0 + decltype(b_)::value;
                    if constexpr (U > 0 && F::kLoad(U)) F::template load<U>(row, o, grp, R[kPerUnit ? U - U0 : 0]);
                });
                const uint32_t use = gc * (SPC / NSS) + static_cast<uint32_t>(P / NSS);
                const bool pending = q > 0 || P >= NSS;  // the step's slots hold earlier units of this tile
                // The units' codes are decoded into registers while the
                // slots' previous MMAs may still run (the pin keeps the
                // decode from moving ahead of the previous step), then the
                // slots are taken over: their old D read out and scaled, the
                // new codes stored and the slots handed to the MMA warps.
                uint32_t av[BATCH][8 * KPW];
                float nsc[BATCH][RPW];
#pragma unroll
                for (int bb = 0; bb < (kPerUnit ? BATCH : 1); ++bb) F::pin(R[bb]);
                static_for<0, BATCH>([&](auto b_) {
                    constexpr int BI = decltype(b_)::value;
                    F::template decode<U0 + BI>(R[kPerUnit ? BI : 0], av[BI], nsc[BI]);
                });
                if constexpr (U0 <= F::kLastLoad && F::kLastLoad < U0 + BATCH) {
                    // the staged weights and inputs of this chunk are all
                    // read, and the words decoded (the release has no load
                    // left to wait for)
                    __syncwarp();
                    if (lane == 0) mbar_arrive(eb + 8 * st);
                }
                if (pending) {
                    if (__all_sync(0xFFFFFFFFu, dseen)) tc_fence_after();
                    else wait_d(SS, use - 1u);
                    if (failed) return;
                }
                if constexpr (P == 0) fseen = more && mbar_test(fb + 8 * st1, ph1);
#pragma unroll
                for (int bb = 0; bb < BATCH; ++bb)
                    tmem_st_cols<KPW>(tmem + lane_base + static_cast<uint32_t>(((U0 + bb) % NS) * G::ACOLS + 8 * KPW * grp),
                                      av[bb]);
                if constexpr (kEarlyD) {
                    if (pending) {
                        if (!dn_ok) {
#pragma unroll
                            for (int bb = 0; bb < BATCH; ++bb) load_d((U0 + bb) % NS, dn[kEarlyD ? bb : 0]);
                        }
                        tmem_ld_wait();
#pragma unroll
                        for (int bb = 0; bb < BATCH; ++bb)
                            tc_scale<MP, RPW>(dn[kEarlyD ? bb : 0], psc[(U0 + bb) % NS], acc);
                    }
                } else {
                    uint32_t d[BATCH][RPW * G::NCOL];
                    if (pending) {
#pragma unroll
                        for (int bb = 0; bb < BATCH; ++bb) load_d((U0 + bb) % NS, d[bb]);
                        tmem_ld_wait();
#pragma unroll
                        for (int bb = 0; bb < BATCH; ++bb) tc_scale<MP, RPW>(d[bb], psc[(U0 + bb) % NS], acc);
                    }
                }
#pragma unroll
                for (int bb = 0; bb < BATCH; ++bb)
#pragma unroll
                    for (int r = 0; r < RPW; ++r) psc[(U0 + bb) % NS][r] = nsc[bb][r];
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(ab + 8 * SS);
                // poll the next step's slot barrier now (its previous use was
                // handed over a step ago); the wait there uses the answer
                if constexpr (!kLast) {
                    constexpr int P1 = P + 1;
                    const uint32_t use1 = gc * (SPC / NSS) + static_cast<uint32_t>(P1 / NSS);
                    const bool pend1 = q > 0 || P1 >= NSS;
                    dseen = pend1 && mbar_test(db + 8 * (P1 % NSS), (use1 - 1u) & 1u);
                } else {
                    const uint32_t use1 = (gc + 1u) * (SPC / NSS);
                    dseen = more && mbar_test(db + 8 * 0, (use1 - 1u) & 1u);
                }
                if constexpr (kEarlyD) {
                    // the next step's slots: (BATCH * P1 + bb) % NS, or the next chunk's first step's
                    constexpr int N0 = kLast ? 0 : BATCH * (P + 1);
                    dn_ok = __all_sync(0xFFFFFFFFu, dseen);
                    if (dn_ok) {
                        tc_fence_after();
#pragma unroll
                        for (int bb = 0; bb < BATCH; ++bb) load_d((N0 + bb) % NS, dn[kEarlyD ? bb : 0]);
                    }
                }
                if constexpr (kLast) {
                    if (more) open_chunk(st1, ph1, q + 1, (gc + 1u) & 1u, R[0], fseen);
                }
            });
            st = st1;
            ph = ph1;
        }
        // drain: the last step of every step slot, in unit order
        if (nck > 0) {
            static_for<0, NSS>([&](auto s_) {
                constexpr int SS = decltype(s_)::value;
                wait_d(SS, (gc - 1u) * (SPC / NSS) + static_cast<uint32_t>((SPC - NSS + SS) / NSS));
                if (failed) return;
                static_for<0, BATCH>([&](auto b_) {
                    constexpr int SL = SS * BATCH + decltype(b_)::value;
                    uint32_t d[RPW * G::NCOL];
                    load_d(SL, d);
                    tmem_ld_wait();
                    tc_scale<MP, RPW>(d, psc[SL], acc);
                });
            });
        }
        // the other warp groups' partials join group 0's, in group order
        float* pb = pairs + (t & 1u) * pair_floats;
        if (grp > 0) {
#pragma unroll
            for (int j = 0; j < MP; ++j)
                pb[((grp - 1) * 4 * MP + quarter * MP + j) * 32 + lane] = failed ? __int_as_float(0x7FC00000) : acc[j];
        }
        asm volatile("bar.sync 2, %0;" ::"n"(CW * 32) : "memory");
        float part[1][MP];
#pragma unroll
        for (int j = 0; j < MP; ++j) {
            float v = failed ? __int_as_float(0x7FC00000) : acc[j];
            if (grp == 0) {
#pragma unroll
                for (int g = 1; g < G::GROUPS; ++g) v = __fadd_rn(v, pb[((g - 1) * 4 * MP + quarter * MP + j) * 32 + lane]);
            }
            part[0][j] = v;
        }
        finish_row_block<1, MP, 32>(part, a, b, wrow0, wrow0 < a.n, lane, 0, lane, quarter, s, S, t, parts,
                                    pair_floats, [&](int j) { return static_cast<uint32_t>(j) < m; }, grp == 0);
    }
    if (S > 1) cluster_sync();
    tmem_ld_wait();  // no read of tensor memory outlives the warp (an early read after a failed wait)
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"n"((CW + 2) * 32) : "memory");
}

}  // namespace dev
}  // namespace rem

// Kernel pointer of rem_tc_kernel<WT, MP, CM>, or nullptr where MP exceeds
// the format's limit or no m of the width MP takes that conversion mode
// (tc_conv_mma).
namespace rem {
template <int WT, int MP, bool CM>
inline const void* tc_kernel_ptr() {
    constexpr uint32_t mlo = static_cast<uint32_t>(MP / 2 + 1), mhi = static_cast<uint32_t>(MP);
    if constexpr (MP > tc_max_mp(WT) || (CM && !tc_conv_mma(WT, mlo)) || (!CM && tc_conv_mma(WT, mhi))) {
        return nullptr;
    } else {
        return reinterpret_cast<const void*>(&dev::rem_tc_kernel<WT, MP, CM>);
    }
}
}  // namespace rem

#define REM_TC_INSTANTIATE(WT, NAME)                                                              \
    namespace rem {                                                                               \
    template <bool CM>                                                                            \
    static const void* NAME##_cm(int mp) {                                                        \
        switch (mp) {                                                                             \
        case 1: return tc_kernel_ptr<WT, 1, CM>();                                                \
        case 2: return tc_kernel_ptr<WT, 2, CM>();                                                \
        case 4: return tc_kernel_ptr<WT, 4, CM>();                                                \
        case 8: return tc_kernel_ptr<WT, 8, CM>();                                                \
        case 16: return tc_kernel_ptr<WT, 16, CM>();                                              \
        case 32: return tc_kernel_ptr<WT, 32, CM>();                                              \
        default: return nullptr;                                                                  \
        }                                                                                         \
    }                                                                                             \
    const void* NAME(int mp, bool cm) { return cm ? NAME##_cm<true>(mp) : NAME##_cm<false>(mp); } \
    }
