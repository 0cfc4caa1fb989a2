// rem_aux.cu -- exact dequantization and round-to-nearest quantization of
// the weight formats of mlx-native 0.18.0 src/ops/row_exact_matvec.rs
// (RowExactWeight: F16, Q8_0, Q4_K, Q6_K, Q5_0) and of the dense F32 / BF16
// weights of the row-independent gemv (nuvec-core 0.6.0 src/gpu.rs), on the GPU.
//
// Every floating-point step is an explicitly rounded intrinsic
// (__fmul_rn, __fsub_rn, __fdiv_rn, __fadd_rn), so the results do not depend
// on contraction or on the compiler: a dequantized value is
//   F16  the binary16 value          Q8_0  d*q          Q5_0  d*(q-16)
//   F32  the binary32 value          BF16  the upper half of a binary32
//   Q4_K (d*sc)*q - dmin*mn          Q6_K  (d*sc)*(q-32)
// and a quantized code is roundf(x / stored_scale), clamped.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "rem_internal.h"

namespace rem {
namespace aux {

__device__ __forceinline__ float h2f(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
}
__device__ __forceinline__ uint32_t rd16(const uint8_t* p) { return p[0] | (static_cast<uint32_t>(p[1]) << 8); }
__device__ __forceinline__ uint32_t rd32(const uint8_t* p) {
    return p[0] | (static_cast<uint32_t>(p[1]) << 8) | (static_cast<uint32_t>(p[2]) << 16) |
           (static_cast<uint32_t>(p[3]) << 24);
}
// Every 16-bit field of every format sits at an even offset of a block, and
// blocks start at even addresses (W is at least 2-byte aligned), so a field
// is written with one aligned 16-bit store.
__device__ __forceinline__ void wr16(uint8_t* p, uint32_t v) {
    *reinterpret_cast<uint16_t*>(p) = static_cast<uint16_t>(v & 0xFFFFu);
}
__device__ __forceinline__ int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }
__device__ __forceinline__ uint32_t h_rn(float f) { return __half_as_ushort(__float2half_rn(f)); }
__device__ __forceinline__ uint32_t h_ru(float f) { return __half_as_ushort(__float2half_ru(f)); }
// binary32 -> bfloat16 bits, round to nearest even on the 16 dropped bits;
// a NaN keeps its upper bits with the quiet bit set.
__device__ __forceinline__ uint32_t bf_rn(float f) {
    const uint32_t u = __float_as_uint(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u) return (u >> 16) | 0x0040u;
    uint32_t keep = u >> 16;
    const uint32_t rest = u & 0xFFFFu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;
    return keep & 0xFFFFu;
}

// ---------------------------------------------------------------- dequantize

// One thread per group of 32 values (a Q8_0 / Q5_0 block, a Q4_K sub-block,
// two Q6_K sub-blocks, or 32 F16 / F32 / BF16 values).
__global__ void dequant_kernel(const uint8_t* __restrict__ w, int wt, uint64_t rows, uint32_t k,
                               uint64_t row_bytes, float* __restrict__ out) {
    const uint64_t groups_per_row = (k + 31u) / 32u;  // F16 rows may end in a partial group
    const uint64_t tid = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (tid >= rows * groups_per_row) return;
    const uint64_t r = tid / groups_per_row;
    const uint32_t gi = static_cast<uint32_t>(tid - r * groups_per_row);
    const uint8_t* row = w + r * row_bytes;
    float* o = out + r * k + 32u * gi;
    if (wt == kF16) {
        const uint32_t nv = min(32u, k - 32u * gi);
        for (uint32_t e = 0; e < nv; ++e) o[e] = h2f(rd16(row + 2u * (32u * gi + e)));
    } else if (wt == kBF16) {
        const uint32_t nv = min(32u, k - 32u * gi);
        for (uint32_t e = 0; e < nv; ++e) o[e] = __uint_as_float(rd16(row + 2u * (32u * gi + e)) << 16);
    } else if (wt == kF32) {
        const uint32_t nv = min(32u, k - 32u * gi);
        for (uint32_t e = 0; e < nv; ++e) o[e] = __uint_as_float(rd32(row + 4u * (32u * gi + e)));
    } else if (wt == kQ8_0) {
        const uint8_t* b = row + 34u * gi;
        const float d = h2f(rd16(b));
        for (int e = 0; e < 32; ++e) o[e] = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(b[2 + e])));
    } else if (wt == kQ5_0) {
        const uint8_t* b = row + 22u * gi;
        const float d = h2f(rd16(b));
        const uint32_t qh = rd32(b + 2);
        for (int e = 0; e < 32; ++e) {
            const int nib = (e < 16) ? (b[6 + e] & 0x0F) : (b[6 + e - 16] >> 4);
            const int q = nib | static_cast<int>(((qh >> e) & 1u) << 4);
            o[e] = __fmul_rn(d, static_cast<float>(q - 16));
        }
    } else if (wt == kQ4_K) {
        const uint8_t* b = row + 144u * (gi / 8u);
        const int s = static_cast<int>(gi % 8u);  // sub-block of 32
        const float d = h2f(rd16(b)), dmin = h2f(rd16(b + 2));
        const uint8_t* sc12 = b + 4;
        int sc, mn;
        if (s < 4) {
            sc = sc12[s] & 63;
            mn = sc12[s + 4] & 63;
        } else {
            sc = (sc12[s + 4] & 0x0F) | ((sc12[s - 4] >> 6) << 4);
            mn = (sc12[s + 4] >> 4) | ((sc12[s] >> 6) << 4);
        }
        const float scale = __fmul_rn(d, static_cast<float>(sc));
        const float minv = __fmul_rn(dmin, static_cast<float>(mn));
        const uint8_t* qs = b + 16 + 32 * (s / 2);
        for (int l = 0; l < 32; ++l) {
            const int q = (s & 1) ? (qs[l] >> 4) : (qs[l] & 0x0F);
            o[l] = __fsub_rn(__fmul_rn(scale, static_cast<float>(q)), minv);
        }
    } else {  // Q6_K: values 32*(gi%8) .. +31 of super-block gi/8
        const uint8_t* b = row + 210u * (gi / 8u);
        const float d = h2f(rd16(b + 208));
        const int e0 = 32 * static_cast<int>(gi % 8u);
        for (int l = 0; l < 32; ++l) {
            const int e = e0 + l;
            const int h = e / 128, t = (e % 128) / 32, ll = e % 32;
            const uint8_t lb = b[64 * h + ll + 32 * (t & 1)];
            const int lo = (t < 2) ? (lb & 0x0F) : (lb >> 4);
            const int hb = (b[128 + 32 * h + ll] >> (2 * t)) & 3;
            const int q = lo | (hb << 4);
            const int sc = static_cast<int8_t>(b[192 + 8 * h + 2 * t + ll / 16]);
            o[l] = __fmul_rn(__fmul_rn(d, static_cast<float>(sc)), static_cast<float>(q - 32));
        }
    }
}

// ---------------------------------------------------------------- quantize

__device__ void quant_q8_0(const float* v, uint8_t* b) {
    float amax = 0.0f;
    for (int e = 0; e < 32; ++e) {
        const float a = fabsf(v[e]);
        if (a > amax) amax = a;
    }
    const uint32_t dh = h_rn(__fdiv_rn(amax, 127.0f));
    const float d = h2f(dh);
    wr16(b, dh);
    for (int e = 0; e < 32; ++e) {
        int q = 0;
        if (d != 0.0f) q = clampi(static_cast<int>(roundf(__fdiv_rn(v[e], d))), -127, 127);
        b[2 + e] = static_cast<uint8_t>(static_cast<int8_t>(q));
    }
}

__device__ void quant_q5_0(const float* v, uint8_t* b) {
    float amax = 0.0f, vmax = 0.0f;
    for (int e = 0; e < 32; ++e) {
        const float a = fabsf(v[e]);
        if (a > amax) {
            amax = a;
            vmax = v[e];
        }
    }
    const uint32_t dh = h_rn(__fdiv_rn(vmax, -16.0f));
    const float d = h2f(dh);
    int q[32];
    for (int e = 0; e < 32; ++e) {
        q[e] = 16;
        if (d != 0.0f) q[e] = clampi(static_cast<int>(roundf(__fdiv_rn(v[e], d))) + 16, 0, 31);
    }
    wr16(b, dh);
    uint32_t qh = 0;
    for (int e = 0; e < 32; ++e) qh |= static_cast<uint32_t>((q[e] >> 4) & 1) << e;
    b[2] = static_cast<uint8_t>(qh);
    b[3] = static_cast<uint8_t>(qh >> 8);
    b[4] = static_cast<uint8_t>(qh >> 16);
    b[5] = static_cast<uint8_t>(qh >> 24);
    for (int i = 0; i < 16; ++i) b[6 + i] = static_cast<uint8_t>((q[i] & 0x0F) | ((q[i + 16] & 0x0F) << 4));
}

__device__ void quant_q4_k(const float* v, uint8_t* b) {
    float lo[8], hi[8];
    for (int s = 0; s < 8; ++s) {
        float mnv = 0.0f, mxv = 0.0f;
        for (int e = 0; e < 32; ++e) {
            const float x = v[32 * s + e];
            if (x < mnv) mnv = x;
            if (x > mxv) mxv = x;
        }
        lo[s] = mnv;
        hi[s] = mxv;
    }
    float mneg = 0.0f;
    for (int s = 0; s < 8; ++s)
        if (-lo[s] > mneg) mneg = -lo[s];
    const uint32_t dminh = h_ru(__fdiv_rn(mneg, 63.0f));
    const float dmin = h2f(dminh);
    int mn[8];
    for (int s = 0; s < 8; ++s) {
        mn[s] = 0;
        if (dmin > 0.0f) mn[s] = clampi(static_cast<int>(ceilf(__fdiv_rn(-lo[s], dmin))), 0, 63);
    }
    float range[8], rmax = 0.0f;
    for (int s = 0; s < 8; ++s) {
        const float off = __fmul_rn(dmin, static_cast<float>(mn[s]));
        range[s] = __fadd_rn(hi[s], off);
        const float r15 = __fdiv_rn(range[s], 15.0f);
        if (r15 > rmax) rmax = r15;
    }
    const uint32_t dh = h_ru(__fdiv_rn(rmax, 63.0f));
    const float d = h2f(dh);
    int sc[8];
    for (int s = 0; s < 8; ++s) {
        sc[s] = 0;
        if (d > 0.0f) sc[s] = clampi(static_cast<int>(ceilf(__fdiv_rn(__fdiv_rn(range[s], 15.0f), d))), 1, 63);
    }
    wr16(b, dh);
    wr16(b + 2, dminh);
    uint8_t* s12 = b + 4;
    for (int s = 0; s < 4; ++s) {
        s12[s] = static_cast<uint8_t>((sc[s] & 63) | ((sc[s + 4] >> 4) << 6));
        s12[s + 4] = static_cast<uint8_t>((mn[s] & 63) | ((mn[s + 4] >> 4) << 6));
        s12[s + 8] = static_cast<uint8_t>((sc[s + 4] & 0x0F) | ((mn[s + 4] & 0x0F) << 4));
    }
    uint8_t* qs = b + 16;
    for (int c = 0; c < 4; ++c) {
        const int s0 = 2 * c, s1 = 2 * c + 1;
        const float off0 = __fmul_rn(dmin, static_cast<float>(mn[s0]));
        const float off1 = __fmul_rn(dmin, static_cast<float>(mn[s1]));
        const float den0 = __fmul_rn(d, static_cast<float>(sc[s0]));
        const float den1 = __fmul_rn(d, static_cast<float>(sc[s1]));
        for (int l = 0; l < 32; ++l) {
            int q0 = 0, q1 = 0;
            if (den0 > 0.0f)
                q0 = clampi(static_cast<int>(roundf(__fdiv_rn(__fadd_rn(v[32 * s0 + l], off0), den0))), 0, 15);
            if (den1 > 0.0f)
                q1 = clampi(static_cast<int>(roundf(__fdiv_rn(__fadd_rn(v[32 * s1 + l], off1), den1))), 0, 15);
            qs[32 * c + l] = static_cast<uint8_t>(q0 | (q1 << 4));
        }
    }
}

__device__ void quant_q6_k(const float* v, uint8_t* b) {
    float amax[16], top = 0.0f;
    for (int s = 0; s < 16; ++s) {
        float a = 0.0f;
        for (int e = 0; e < 16; ++e) {
            const float t = fabsf(v[16 * s + e]);
            if (t > a) a = t;
        }
        amax[s] = a;
        if (a > top) top = a;
    }
    const uint32_t dh = h_ru(__fdiv_rn(top, 3937.0f));  // 31 * 127
    const float d = h2f(dh);
    const float d31 = __fmul_rn(31.0f, d);
    int sc[16];
    for (int s = 0; s < 16; ++s) {
        sc[s] = 0;
        if (d > 0.0f) sc[s] = clampi(static_cast<int>(ceilf(__fdiv_rn(amax[s], d31))), 0, 127);
    }
    for (int i = 0; i < 192; ++i) b[i] = 0;
    for (int s = 0; s < 16; ++s) {
        const float den = __fmul_rn(d, static_cast<float>(sc[s]));
        for (int l16 = 0; l16 < 16; ++l16) {
            const int e = 16 * s + l16;
            int q = 32;
            if (den > 0.0f) q = clampi(static_cast<int>(roundf(__fdiv_rn(v[e], den))) + 32, 0, 63);
            const int h = e / 128, t = (e % 128) / 32, l = e % 32;
            const int lo = q & 0x0F, hb = q >> 4;
            b[64 * h + l + 32 * (t & 1)] |= static_cast<uint8_t>(t < 2 ? lo : (lo << 4));
            b[128 + 32 * h + l] |= static_cast<uint8_t>(hb << (2 * t));
        }
    }
    for (int s = 0; s < 16; ++s) b[192 + s] = static_cast<uint8_t>(static_cast<int8_t>(sc[s]));
    wr16(b + 208, dh);
}

// One thread per block (per value for F16, F32 and BF16).
__global__ void quant_kernel(const float* __restrict__ src, int wt, uint64_t rows, uint32_t k, uint64_t row_bytes,
                             uint8_t* __restrict__ w) {
    const uint32_t bv = static_cast<uint32_t>(block_values(wt));
    const uint64_t per_row = k / bv;
    const uint64_t tid = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (tid >= rows * per_row) return;
    const uint64_t r = tid / per_row;
    const uint32_t bi = static_cast<uint32_t>(tid - r * per_row);
    const float* v = src + r * k + static_cast<uint64_t>(bi) * bv;
    uint8_t* b = w + r * row_bytes + static_cast<uint64_t>(bi) * block_bytes(wt);
    switch (wt) {
    case kF16: wr16(b, h_rn(v[0])); break;
    case kBF16: wr16(b, bf_rn(v[0])); break;
    case kF32: *reinterpret_cast<uint32_t*>(b) = __float_as_uint(v[0]); break;
    case kQ8_0: quant_q8_0(v, b); break;
    case kQ5_0: quant_q5_0(v, b); break;
    case kQ4_K: quant_q4_k(v, b); break;
    default: quant_q6_k(v, b); break;
    }
}

// Affine: one thread per group; w = fl(fl(scale * q) + bias); a row's codes
// are one little-endian bit stream, code i at bits [bits*i, bits*i + bits).
__global__ void dequant_affine_kernel(const uint32_t* __restrict__ codes, const uint16_t* __restrict__ scales,
                                      const uint16_t* __restrict__ biases, int bits, int gs, uint64_t rows,
                                      uint32_t k, float* __restrict__ out) {
    const uint64_t ng = k / static_cast<uint32_t>(gs);
    const uint64_t tid = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (tid >= rows * ng) return;
    const uint64_t r = tid / ng, g = tid - r * ng;
    const uint32_t mask = (1u << bits) - 1u;
    const uint64_t nbytes = static_cast<uint64_t>(k) * bits / 8u;
    const uint8_t* cb = reinterpret_cast<const uint8_t*>(codes) + r * nbytes;
    const float sc = h2f(scales[tid]), bi = h2f(biases[tid]);
    for (int e = 0; e < gs; ++e) {
        const uint64_t i = g * gs + e, bit = i * static_cast<uint64_t>(bits);
        uint32_t v = cb[bit / 8];
        if (bit / 8 + 1 < nbytes) v |= static_cast<uint32_t>(cb[bit / 8 + 1]) << 8;
        const uint32_t q = (v >> (bit % 8)) & mask;
        out[r * k + i] = __fadd_rn(__fmul_rn(sc, static_cast<float>(q)), bi);
    }
}

}  // namespace aux

int launch_dequantize_affine(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases, int wt,
                             uint64_t rows, uint32_t k, float* out, void* stream) {
    const uint64_t threads = rows * (k / static_cast<uint32_t>(affine_group(wt)));
    if (threads == 0) return 0;
    const uint32_t block = 128;
    const uint64_t grid = (threads + block - 1) / block;
    aux::dequant_affine_kernel<<<static_cast<unsigned>(grid), block, 0, static_cast<cudaStream_t>(stream)>>>(
        codes, scales, biases, affine_bits(wt), affine_group(wt), rows, k, out);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_dequantize(const uint8_t* w, int wt, uint64_t rows, uint32_t k, uint64_t row_bytes, float* out,
                      void* stream) {
    const uint64_t threads = rows * ((k + 31u) / 32u);
    if (threads == 0) return 0;
    const uint32_t block = 128;
    const uint64_t grid = (threads + block - 1) / block;
    aux::dequant_kernel<<<static_cast<unsigned>(grid), block, 0, static_cast<cudaStream_t>(stream)>>>(
        w, wt, rows, k, row_bytes, out);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_quantize(const float* src, int wt, uint64_t rows, uint32_t k, uint64_t row_bytes, uint8_t* w,
                    void* stream) {
    const uint64_t threads = rows * (k / static_cast<uint32_t>(block_values(wt)));
    if (threads == 0) return 0;
    const uint32_t block = 128;
    const uint64_t grid = (threads + block - 1) / block;
    aux::quant_kernel<<<static_cast<unsigned>(grid), block, 0, static_cast<cudaStream_t>(stream)>>>(
        src, wt, rows, k, row_bytes, w);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace rem
